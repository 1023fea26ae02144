"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import build as BUILD


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.lib()


def header_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"CSA_API\s+[\w\s\*]+?\b(csa_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.EXPORTS)


def test_every_declaration_cites_its_passage():
    """Each entry point's comment cites the page passage it follows, or says the
    pages have no counterpart (workspace queries, status and accounting)."""
    text = open(os.path.join(ROOT, "include", "csa.h")).read()
    decls = list(re.finditer(r"CSA_API\s+[\w\s\*]+?\b(csa_\w+)\s*\(", text))
    assert len(decls) == len(B.EXPORTS)
    for m in decls:
        before = text[:m.start()]
        comment = before[before.rfind("/*"):before.rfind("*/") + 2]
        assert "CSA_API" not in before[before.rfind("*/"):], (m.group(1), "no comment of its own")
        squashed = " ".join(comment.replace("*", " ").split())
        assert any(k in squashed for k in ("G2C Brief", "Pushing the Limits", "no counterpart", "No counterpart",
                                           "describe no counterpart")), m.group(1)


def test_status_strings(lib):
    for s in range(6):
        assert B.status_string(s)
    assert B.status_string(0) == "ok"


def fake_cache(**kw):
    # 16-byte aligned fake device addresses: only checked, never dereferenced.
    d = dict(batch=2, capacity=64, d_latent=128, d_index=64, codes=0x10000, scales=0x20000, ikeys=0x30000,
             lengths=0x40000)
    d.update(kw)
    return B.csa_cache(**d)


def test_null_and_bad_cache_rejected_before_launch(lib):
    assert lib.csa_quantize_append(None, None, None, 1, None) == 1
    c = fake_cache(d_latent=100)
    assert lib.csa_quantize_append(ctypes.byref(c), ctypes.c_void_p(0x50000), None, 1, None) == 1
    c = fake_cache(d_latent=1024)
    assert lib.csa_quantize_append(ctypes.byref(c), ctypes.c_void_p(0x50000), None, 1, None) == 2
    c = fake_cache(codes=0x10008)                                     # misaligned
    assert lib.csa_quantize_append(ctypes.byref(c), ctypes.c_void_p(0x50000), None, 1, None) == 1
    c = fake_cache()
    assert lib.csa_quantize_append(ctypes.byref(c), ctypes.c_void_p(0x50000), None, -1, None) == 1
    big = fake_cache(batch=2, capacity=1 << 30)                       # 2^31 rows: 32-bit row ids overflow
    assert lib.csa_quantize_append(ctypes.byref(big), ctypes.c_void_p(0x50000), None, 1, None) == 2
    assert lib.csa_cache_record_bytes(ctypes.byref(big)) == 0
    assert lib.csa_quantize_append(ctypes.byref(c), ctypes.c_void_p(0x50000), None, 0, None) == 0


def test_argument_checks_of_each_call(lib):
    c = ctypes.byref(fake_cache())
    V = ctypes.c_void_p
    # index score: ld below capacity, HI*P too large
    assert lib.csa_index_score(c, 1, 4, V(0x1000), V(0x2000), None, 0, V(0x3000), 32, None, 0, None) == 1
    assert lib.csa_index_score(c, 8, 128, V(0x1000), V(0x2000), None, 0, V(0x3000), 64, None, 0, None) == 2
    # block maxima (capacity 64: 8 blocks): with a pool, a stride below 8 or not a
    # multiple of 4, a misaligned buffer
    assert lib.csa_index_score(c, 1, 4, V(0x1000), V(0x2000), V(0x4000), 4, V(0x3000), 64, V(0x5000), 8, None) == 1
    assert lib.csa_index_score(c, 1, 4, V(0x1000), V(0x2000), None, 0, V(0x3000), 64, V(0x5000), 4, None) == 1
    assert lib.csa_index_score(c, 1, 4, V(0x1000), V(0x2000), None, 0, V(0x3000), 64, V(0x5000), 10, None) == 1
    assert lib.csa_index_score(c, 1, 4, V(0x1000), V(0x2000), None, 0, V(0x3000), 64, V(0x5008), 8, None) == 1
    # top-K: K out of range; pool_out together with a pool
    assert lib.csa_topk(c, 1, V(0x1000), 64, None, 0, 0, V(0x2000), 0, None, None, 0, None, 0, None) == 1
    assert lib.csa_topk(c, 1, V(0x1000), 64, V(0x4000), 8, 4, V(0x2000), 8, V(0x5000), None, 0, None, 0, None) == 1
    # block maxima without a pool to build, or with a stride below 8
    assert lib.csa_topk(c, 1, V(0x1000), 64, None, 0, 4, V(0x2000), 0, None, V(0x6000), 8, None, 0, None) == 1
    assert lib.csa_topk(c, 1, V(0x1000), 64, None, 0, 4, V(0x2000), 4, V(0x5000), V(0x6000), 4, None, 0, None) == 1
    # a row longer than one cluster holds is selected in two stages through the workspace
    n = ctypes.c_size_t(0)
    big = ctypes.byref(fake_cache(capacity=1 << 20))
    assert lib.csa_topk_workspace_size(big, 1, 0, 2048, 0, ctypes.byref(n)) == 0 and n.value > 0
    assert lib.csa_topk(big, 1, V(0x1000), 1 << 20, None, 0, 2048, V(0x2000), 0, None, None, 0, None, 0, None) == 5
    assert lib.csa_topk_workspace_size(c, 1, 0, 2048, 0, ctypes.byref(n)) == 0 and n.value == 0
    # attention: too many heads, missing workspace
    assert lib.csa_sparse_attend(c, 1, 65, V(0x1000), 1.0, V(0x2000), 8, V(0x3000), None, V(0x4000), 1 << 20,
                                 None) == 2
    # K=2048 over 2 queries is split over several CTAs whose partials meet in
    # the workspace: a call without one is refused before any launch
    assert lib.csa_sparse_attend(c, 1, 16, V(0x1000), 1.0, V(0x2000), 2048, V(0x3000), None, None, 0, None) == 5
    n = ctypes.c_size_t(0)
    assert lib.csa_attend_workspace_size(c, 1, 16, 2048, ctypes.byref(n)) == 0 and n.value > 0
    # with a local window (K=2048 over 2 queries), the splits' partials go through
    # the workspace, and a call without one is refused before any launch
    win = B.csa_swa(rows=0x7000, lengths=None, n=128, window=128)
    assert lib.csa_attend_swa_workspace_size(c, 1, 16, 2048, ctypes.byref(win), ctypes.byref(n)) == 0
    assert n.value > 0
    assert lib.csa_sparse_attend_swa(c, 1, 16, V(0x1000), 1.0, V(0x2000), 2048, ctypes.byref(win), V(0x3000), None,
                                     None, 0, None) == 5
    # the spread form of the pool's one-call top-K: its keys need pool_blocks * 8
    # words per query; a shorter workspace is refused before any launch
    c128 = ctypes.byref(fake_cache(d_index=128))
    assert lib.csa_pool_topk_workspace_size(c128, 1, 300, ctypes.byref(n)) == 0 and n.value == 2 * 300 * 8 * 4
    assert lib.csa_pool_topk(c128, 1, 64, V(0x1000), V(0x2000), V(0x3000), 300, 700, V(0x4000), V(0x5000),
                             n.value - 16, None) == 5
    assert lib.csa_pool_topk(c128, 1, 64, V(0x1000), V(0x2000), V(0x3000), 300, 700, V(0x4000), V(0x5008),
                             n.value, None) == 5


def test_layer_args_checks(lib):
    c = ctypes.byref(fake_cache())
    a = B.csa_layer_args(mode=7, P=1, H=16, HI=4, K=8, scale=1.0, q=0x1000, iq=0x2000, w=0x3000, idx=0x4000,
                         out=0x5000)
    n = ctypes.c_size_t(0)
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 1
    a.mode = B.CSA_REUSE
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 0
    reuse_bytes = n.value
    a.mode = B.CSA_FULL
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value >= reuse_bytes + 2 * 64 * 4                      # + scores [B][P][capacity]
    a.pool_in = 0x6000                                              # a pool is a Reindex input only
    a.pool_blocks = 4
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 1
    a.mode = B.CSA_REUSE
    a.pool_in = None
    a.n_new = 2                                                     # only Full appends
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 1
    # workspace missing -> rejected before launch
    a.mode, a.n_new = B.CSA_FULL, 0
    assert lib.csa_layer_step(c, ctypes.byref(a), None) == 5


def test_local_window_checks(lib):
    c = ctypes.byref(fake_cache())
    V = ctypes.c_void_p
    n = ctypes.c_size_t(0)
    ok = B.csa_swa(rows=0x7000, lengths=None, n=128, window=128)
    assert lib.csa_attend_swa_workspace_size(c, 1, 16, 8, ctypes.byref(ok), ctypes.byref(n)) == 0
    for bad in (B.csa_swa(rows=None, lengths=None, n=128, window=128),     # no rows
                B.csa_swa(rows=0x7008, lengths=None, n=128, window=128),   # misaligned rows
                B.csa_swa(rows=0x7000, lengths=None, n=0, window=128),     # fewer rows than positions
                B.csa_swa(rows=0x7000, lengths=None, n=128, window=0),     # empty window
                B.csa_swa(rows=0x7000, lengths=None, n=2048, window=1025)):
        assert lib.csa_attend_swa_workspace_size(c, 1, 16, 8, ctypes.byref(bad), ctypes.byref(n)) == 1
        assert lib.csa_sparse_attend_swa(c, 1, 16, V(0x1000), 1.0, V(0x2000), 8, ctypes.byref(bad), V(0x3000),
                                         None, V(0x4000), 1 << 20, None) == 1
    # no window: the same sizes as csa_attend_workspace_size
    m = ctypes.c_size_t(0)
    assert lib.csa_attend_swa_workspace_size(c, 1, 16, 2048, None, ctypes.byref(n)) == 0
    assert lib.csa_attend_workspace_size(c, 1, 16, 2048, ctypes.byref(m)) == 0 and m.value == n.value
    # with a window, 2 queries still split over more CTAs than a cluster holds
    assert lib.csa_attend_swa_workspace_size(c, 1, 16, 2048, ctypes.byref(ok), ctypes.byref(n)) == 0
    assert n.value > 0
    # a layer step validates its window too
    a = B.csa_layer_args(mode=B.CSA_REUSE, P=2, H=16, K=8, scale=1.0, q=0x1000, idx=0x4000, out=0x5000)
    bad = B.csa_swa(rows=0x7000, lengths=None, n=1, window=8)
    a.swa = ctypes.addressof(bad)
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 1
    good = B.csa_swa(rows=0x7000, lengths=None, n=4, window=8)
    a.swa = ctypes.addressof(good)
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 0


def test_projected_append_checks(lib):
    c = ctypes.byref(fake_cache())
    V = ctypes.c_void_p
    assert lib.csa_quantize_append_project(c, V(0x50000), None, 1, None) == 1            # no matrix
    assert lib.csa_quantize_append_project(c, V(0x50000), V(0x60008), 1, None) == 1      # misaligned matrix
    assert lib.csa_quantize_append_project(ctypes.byref(fake_cache(d_index=48)), V(0x50000), V(0x60000), 1,
                                           None) == 2                                     # d_index not 32/64/128
    assert lib.csa_quantize_append_project(c, V(0x50000), V(0x60000), 0, None) == 0       # nothing to append
    a = B.csa_layer_args(mode=B.CSA_FULL, P=1, H=16, HI=4, K=8, scale=1.0, q=0x1000, iq=0x2000, w=0x3000,
                         idx=0x4000, out=0x5000, rows_new=0x7000, ikeys_new=0x8000, n_new=1, w_ik=0x9000)
    n = ctypes.c_size_t(0)
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 1        # keys given and projected
    a.ikeys_new = None
    assert lib.csa_layer_workspace_size(c, ctypes.byref(a), ctypes.byref(n)) == 0


def test_mxfp4_cache_checks(lib):
    V = ctypes.c_void_p
    ok = dict(d_index=128, ikey_format=B.CSA_IKEY_MXFP4, iscales=0x60000)
    assert lib.csa_quantize_append(ctypes.byref(fake_cache(**ok)), V(0x50000), None, 0, None) == 0
    bad = [
        (dict(ok, ikey_format=7), 1),                 # unknown key format
        (dict(ok, iscales=None), 1),                  # no block scales
        (dict(ok, iscales=0x60008), 1),               # misaligned scales
        (dict(ok, ikeys=0x30010), 1),                 # keys 16- but not 32-byte aligned
        (dict(ok, d_index=64), 2),                    # MXFP4 keys are 128 channels
        (dict(ok, capacity=62), 2),                   # capacity a multiple of 4
    ]
    for kw, want in bad:
        assert lib.csa_quantize_append(ctypes.byref(fake_cache(**kw)), V(0x50000), None, 0, None) == want, kw


def test_persistent_record_checks(lib):
    V = ctypes.c_void_p
    lib.csa_cache_record_bytes.restype = ctypes.c_size_t
    c = fake_cache()                                                        # D 128, d_index 64, E4M3
    assert lib.csa_cache_record_bytes(ctypes.byref(c)) == 64 + 8 + 64
    mx = fake_cache(d_index=128, ikey_format=B.CSA_IKEY_MXFP4, iscales=0x60000)
    assert lib.csa_cache_record_bytes(ctypes.byref(mx)) == 64 + 8 + 64 + 4
    big = fake_cache(d_latent=512, d_index=128, ikey_format=B.CSA_IKEY_MXFP4, iscales=0x60000)
    assert lib.csa_cache_record_bytes(ctypes.byref(big)) == 356            # the 288 + 68 B entry
    assert lib.csa_cache_record_bytes(None) == 0
    r = ctypes.byref(c)
    assert lib.csa_cache_spill(r, 0, 0, None, None) == 0                    # nothing to spill
    assert lib.csa_cache_spill(r, -1, 4, V(0x70000), None) == 1
    assert lib.csa_cache_spill(r, 60, 5, V(0x70000), None) == 1             # past capacity 64
    assert lib.csa_cache_spill(r, 0, 4, V(0x70002), None) == 1             # misaligned records
    assert lib.csa_cache_spill(r, 0, 4, None, None) == 1
    assert lib.csa_cache_reload(r, V(0x70000), 0, None) == 0
    assert lib.csa_cache_reload(r, V(0x70000), 65, None) == 1               # more than capacity
    assert lib.csa_cache_reload(r, V(0x70001), 4, None) == 1
    assert lib.csa_cache_reload(r, None, 4, None) == 1
    assert lib.csa_cache_reload(None, V(0x70000), 4, None) == 1


def test_binding_constants_match_the_header():
    """Every constant the binding mirrors has the header's value (the no-alloc
    scratch size, the pool block, the device status bits, the key formats)."""
    text = open(os.path.join(ROOT, "include", "csa.h")).read()
    defines = dict(re.findall(r"#define\s+(CSA_[A-Z0-9_]+)\s+([0-9xXa-fA-Fu<>() ]+?)\s*(?:/\*|\n)", text))
    mirrored = ["CSA_NOALLOC_SCRATCH_BYTES", "CSA_POOL_BLOCK", "CSA_DEV_BAD_INDEX", "CSA_DEV_CAPACITY",
                "CSA_DEV_TIMEOUT", "CSA_IKEY_E4M3", "CSA_IKEY_MXFP4"]
    for name in mirrored:
        expr = defines[name].replace("u", "")
        assert re.fullmatch(r"[0-9xXa-fA-F<>() ]+", expr), (name, expr)
        assert eval(expr) == getattr(B, name), (name, expr, getattr(B, name))
