"""Persistent cache records on the GPU (csa_cache_spill / csa_cache_reload)
against the oracle, byte for byte.

"G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache entries, and why
they're safe": a cache entry is its 288-byte main entry and its indexer entry
(68 B in MXFP4), kept in device memory and spilled to host memory or storage.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import device_cache, need_gpu

pytestmark = pytest.mark.gpu

CASES = [("e4m3", 512, 128), ("mxfp4", 512, 128), ("e4m3", 128, 32), ("mxfp4", 256, 128)]


def host_copy(cache):
    """The device cache as the oracle's host cache (keys packed as records store them)."""
    o = oracle.Cache(cache.batch, cache.capacity, cache.d_latent, cache.d_index, cache.key_format)
    o.codes[:] = cache.codes.cpu().numpy()
    o.scales[:] = cache.scales.cpu().numpy()
    o.ikeys[:] = cache.packed_keys().cpu().numpy() if cache.key_format == "mxfp4" else cache.ikeys.cpu().numpy()
    o.lengths[:] = cache.lengths.cpu().numpy()
    return o


def ragged_cache(key_format, D, DI, seed, lengths, cap):
    wl = W.Workload("t", B=len(lengths), L=max(lengths), H=4, D=D, HI=4, DI=DI, K=8, key_format=key_format)
    cache, _, _ = device_cache(wl.scaled(L=max(lengths)), seed)
    if cap != wl.capacity:   # a larger cache with the same rows
        big = B.Cache(wl.B, cap, D, DI, device="cuda", key_format=key_format)
        B.csa_cache_reload(big, B.csa_cache_spill(cache, 0, wl.L))
        cache = big
    cache.lengths.copy_(torch.tensor(lengths, dtype=torch.int32))
    torch.cuda.synchronize()
    return cache


@pytest.mark.parametrize("key_format,D,DI", CASES)
def test_spill_matches_oracle(key_format, D, DI):
    need_gpu()
    lengths = [300, 41, 0, 257]
    cache = ragged_cache(key_format, D, DI, 81, lengths, 300)
    o = host_copy(cache)
    assert B.csa_cache_record_bytes(cache) == oracle.record_bytes(D, DI, key_format)
    for row0, n in [(0, 300), (0, 1), (37, 200), (255, 45), (299, 1)]:
        got = B.csa_cache_spill(cache, row0, n)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), oracle.cache_spill(o, row0, n)), (row0, n)
    # into pinned host memory: the same bytes
    host = torch.empty((len(lengths), 300, B.csa_cache_record_bytes(cache)), dtype=torch.uint8).pin_memory()
    host.fill_(0xA5)
    B.csa_cache_spill(cache, 0, 300, records=host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), oracle.cache_spill(o, 0, 300))
    assert B.csa_device_status() == 0


@pytest.mark.parametrize("key_format,D,DI", CASES)
def test_reload_matches_oracle(key_format, D, DI):
    need_gpu()
    lengths = [10, 0, 32]
    cache = ragged_cache(key_format, D, DI, 82, lengths, 64)
    o = host_copy(cache)
    rb = B.csa_cache_record_bytes(cache)
    recs = W.random_ints((len(lengths), 20, rb), 0, 256, seed=83).to(torch.uint8)
    B.csa_device_status()
    B.csa_cache_reload(cache, recs.cuda())
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    assert oracle.cache_reload(o, recs.numpy()) == 0
    h = host_copy(cache)
    for t in ("codes", "scales", "ikeys", "lengths"):
        assert np.array_equal(getattr(h, t), getattr(o, t)), t
    # from pinned host memory, a second append after the first
    pinned = W.random_ints((len(lengths), 5, rb), 0, 256, seed=84).to(torch.uint8).pin_memory()
    B.csa_cache_reload(cache, pinned)
    torch.cuda.synchronize()
    oracle.cache_reload(o, pinned.numpy())
    h = host_copy(cache)
    for t in ("codes", "scales", "ikeys", "lengths"):
        assert np.array_equal(getattr(h, t), getattr(o, t)), t


def test_reload_past_capacity_leaves_the_sequence_unchanged():
    need_gpu()
    cache = ragged_cache("mxfp4", 128, 128, 85, [8, 8, 8], 12)
    cache.lengths[1] = 10
    torch.cuda.synchronize()
    before = host_copy(cache)
    rb = B.csa_cache_record_bytes(cache)
    recs = torch.full((3, 3, rb), 0x5A, dtype=torch.uint8, device="cuda")
    B.csa_device_status()
    B.csa_cache_reload(cache, recs)
    torch.cuda.synchronize()
    assert B.csa_device_status() & B.CSA_DEV_CAPACITY
    h = host_copy(cache)
    assert list(h.lengths) == [11, 10, 11]
    assert np.array_equal(h.codes[1], before.codes[1]) and np.array_equal(h.ikeys[1], before.ikeys[1])
    assert (h.codes[0, 8:11] == 0x5A).all() and (h.ikeys[2, 8:11] == 0x5A).all()


@pytest.mark.parametrize("key_format", ["e4m3", "mxfp4"])
def test_round_trip_scores_the_same(key_format):
    """Spill a cache to pinned host memory, reload it into an empty cache: the
    cache is the same, and so are its index scores."""
    need_gpu()
    wl = W.Workload("t", B=3, L=2500, H=4, D=512, HI=64, DI=128, K=8, key_format=key_format)
    cache, _, _ = device_cache(wl, 86)
    host = torch.empty((wl.B, wl.L, B.csa_cache_record_bytes(cache)), dtype=torch.uint8).pin_memory()
    B.csa_cache_spill(cache, 0, wl.L, records=host)
    back = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device="cuda", key_format=key_format)
    B.csa_cache_reload(back, host)
    inp = W.layer_inputs(wl, 86, 0, device="cuda")
    s0 = B.csa_index_score(cache, inp["iq"], inp["w"])
    s1 = B.csa_index_score(back, inp["iq"], inp["w"])
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    for t in ("codes", "scales", "ikeys", "lengths"):
        assert torch.equal(getattr(back, t), getattr(cache, t)), t
    if key_format == "mxfp4":
        assert torch.equal(back.iscales, cache.iscales)
    assert torch.equal(s0, s1)


@pytest.mark.slow
def test_full_size_1m_round_trip():
    """One sequence of 1,048,576 MXFP4 entries (373 MB of records) through pinned
    host memory and back; spilled records checked against the oracle on samples."""
    need_gpu()
    wl = W.Workload("t", B=1, L=1 << 20, H=64, D=512, HI=64, DI=128, K=2048, key_format="mxfp4")
    cache, _, _ = device_cache(wl, 87)
    rb = B.csa_cache_record_bytes(cache)
    assert rb == 356
    host = torch.empty((1, wl.L, rb), dtype=torch.uint8).pin_memory()
    B.csa_cache_spill(cache, 0, wl.L, records=host)
    back = B.Cache(1, wl.capacity, wl.D, wl.DI, device="cuda", key_format="mxfp4")
    B.csa_cache_reload(back, host)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    for t in ("codes", "scales", "ikeys", "iscales", "lengths"):
        assert torch.equal(getattr(back, t), getattr(cache, t)), t
    rows = np.sort(W.random_ints((64,), 0, wl.L, seed=88).numpy())
    o = oracle.Cache(1, 1, wl.D, wl.DI, "mxfp4")
    keys = cache.packed_keys()[0].cpu().numpy()
    for r in rows:
        o.codes[0, 0] = cache.codes[0, r].cpu().numpy()
        o.scales[0, 0] = cache.scales[0, r].cpu().numpy()
        o.ikeys[0, 0] = keys[r]
        o.lengths[0] = 1
        assert np.array_equal(host[0, r].numpy(), oracle.cache_spill(o, 0, 1)[0, 0]), r
