"""The binding's guards, on the CPU: the C ABI sees only pointers, so the binding
refuses a tensor smaller than the bytes a call touches, or whose batch or last
dim disagrees with the cache where outputs are shaped from it, before any call
into the library.  Tensors of the right size pass the guards and then stop at
the CUDA-device check (these tests run without a GPU)."""
import pytest
import torch

from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import build as BUILD


@pytest.fixture(scope="module", autouse=True)
def built():
    BUILD.build()
    B.lib()


def cache(key_format="e4m3"):
    return B.Cache(2, 64, 256, 64 if key_format == "e4m3" else 128, device="cpu", key_format=key_format)


def guard_error(fn):
    with pytest.raises(ValueError) as e:
        fn()
    return str(e.value)


def passes_guards(fn):
    # the first check after the guards: the tensors are not CUDA tensors
    assert "expected a CUDA tensor" in guard_error(fn)


def i16(*shape):
    return torch.zeros(shape, dtype=torch.int16)


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def test_append_sizes():
    c = cache()
    assert "rows holds" in guard_error(lambda: B.csa_quantize_append(c, i16(1, 4, 256)))
    assert "ikeys_new holds" in guard_error(lambda: B.csa_quantize_append(c, i16(2, 4, 256), u8(2, 4, 32)))
    passes_guards(lambda: B.csa_quantize_append(c, i16(2, 4, 256), u8(2, 4, 64)))
    mx = cache("mxfp4")
    # MXFP4 key rows are 64 code bytes and 4 scale bytes
    assert "ikeys_new holds" in guard_error(lambda: B.csa_quantize_append(mx, i16(2, 4, 256), u8(2, 4, 64)))
    passes_guards(lambda: B.csa_quantize_append(mx, i16(2, 4, 256), u8(2, 4, 68)))
    assert "w_ik holds" in guard_error(lambda: B.csa_quantize_append_project(c, i16(2, 4, 256), i16(128, 64)))
    passes_guards(lambda: B.csa_quantize_append_project(c, i16(2, 4, 256), i16(256, 64)))


def test_record_sizes():
    c = cache()
    rb = B.csa_cache_record_bytes(c)
    assert rb == 128 + 16 + 64
    assert "records holds" in guard_error(lambda: B.csa_cache_spill(c, 0, 10, records=u8(2, 9, rb)))
    assert "records holds" in guard_error(lambda: B.csa_cache_reload(c, u8(1, 10, rb)))


def test_index_and_topk_shapes():
    c = cache()
    assert "iq has shape" in guard_error(lambda: B.csa_index_score(c, u8(1, 1, 4, 64), f32(1, 1, 4)))
    assert "iq has shape" in guard_error(lambda: B.csa_index_score(c, u8(2, 1, 4, 32), f32(2, 1, 4)))
    assert "w holds" in guard_error(lambda: B.csa_index_score(c, u8(2, 1, 4, 64), f32(2, 1, 3)))
    assert "pool holds" in guard_error(lambda: B.csa_index_score(c, u8(2, 1, 4, 64), f32(2, 1, 4), pool=i32(1, 1, 10)))
    passes_guards(lambda: B.csa_index_score(c, u8(2, 1, 4, 64), f32(2, 1, 4)))
    assert "scores has shape" in guard_error(lambda: B.csa_topk(c, f32(1, 1, 64), 8))
    assert "pool holds" in guard_error(lambda: B.csa_topk(c, f32(2, 1, 80), 8, pool=i32(2, 1, 5)[:1]))
    passes_guards(lambda: B.csa_topk(c, f32(2, 1, 64), 8))


def test_attention_shapes():
    c = cache()
    q = i16(2, 1, 8, 256)
    assert "q has shape" in guard_error(lambda: B.csa_sparse_attend(c, i16(1, 1, 8, 256), i32(1, 1, 16), 0.1))
    assert "q has shape" in guard_error(lambda: B.csa_sparse_attend(c, i16(2, 1, 8, 128), i32(2, 1, 16), 0.1))
    assert "idx holds" in guard_error(lambda: B.csa_sparse_attend(c, q, i32(1, 1, 16), 0.1))
    assert "out holds" in guard_error(lambda: B.csa_sparse_attend(c, q, i32(2, 1, 16), 0.1, out=f32(2, 1, 8, 128)))
    assert "lse holds" in guard_error(lambda: B.csa_sparse_attend_noalloc(c, q, i32(2, 1, 16), 0.1,
                                                                          f32(2, 1, 8, 256), f32(2, 1, 4)))
    passes_guards(lambda: B.csa_sparse_attend(c, q, i32(2, 1, 16), 0.1))
    swa_short = B.Swa.__new__(B.Swa)
    swa_short.rows, swa_short.lengths, swa_short.window = u8(1, 40, 256), None, 16
    swa_short._struct = B.csa_swa(None, None, 40, 16)
    assert "swa rows holds" in guard_error(lambda: B.csa_sparse_attend_swa(c, q, i32(2, 1, 16), 0.1, swa_short))


def test_layer_args_sizes():
    c = cache()
    q = i16(2, 2, 8, 256)
    iq, w = u8(2, 2, 4, 64), f32(2, 2, 4)
    assert "iq holds" in guard_error(lambda: B.LayerArgs(c, B.CSA_FULL, q, 16, 0.1, iq=u8(2, 1, 4, 64), w=w))
    assert "rows_new holds" in guard_error(lambda: B.LayerArgs(c, B.CSA_FULL, q, 16, 0.1, iq=iq, w=w,
                                                                rows_new=i16(1, 3, 256)))
    assert "pool_in holds" in guard_error(lambda: B.LayerArgs(c, B.CSA_REINDEX, q, 16, 0.1, iq=iq, w=w,
                                                               pool_in=i32(2, 2, 10), pool_blocks=16))
    assert "idx holds" in guard_error(lambda: B.LayerArgs(c, B.CSA_REUSE, q, 16, 0.1, idx=i32(2, 2, 8)))
    passes_guards(lambda: B.LayerArgs(c, B.CSA_FULL, q, 16, 0.1, iq=iq, w=w))
