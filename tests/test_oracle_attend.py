"""Pins of the oracle's sparse attention (a5/a6) and of the mode chain (a7)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import workloads as W

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def dequant_ref(codes, scales):
    """Dequantise with a literal E2M1 table and torch's E4M3 cast (independent
    of the oracle's decoders)."""
    c = np.asarray(codes)
    lo, hi = c & 0xF, c >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,))
    mag = GRID[nib & 7]
    val = np.where(nib & 8, -mag, mag)
    s = torch.as_tensor(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return val * np.repeat(s, 16, axis=-1)


def bf16_ref(bits):
    return torch.as_tensor(np.ascontiguousarray(bits)).view(torch.bfloat16).to(torch.float64).numpy()


def small_cache(n, D, seed, std=1.0):
    x = W.random_bf16_bits((n, D), seed, 10, std=std).numpy().view(np.uint16)
    codes, scales = oracle.quantize_rows(x)
    return codes, scales


def test_dequant_matches_independent_table():
    codes, scales = small_cache(40, 64, seed=1, std=3.0)
    assert np.array_equal(oracle.dequantize_rows(codes, scales), dequant_ref(codes, scales))


@pytest.mark.parametrize("D,H", [(64, 3), (128, 16)])
def test_all_rows_selected_equals_dense_attention(D, H):
    """Sparse attention with K = context length is dense softmax attention."""
    n = 97
    codes, scales = small_cache(n, D, seed=2)
    q = W.random_bf16_bits((H, D), 3, 11).numpy().view(np.uint16)
    scale = 1.0 / np.sqrt(D)
    out, lse = oracle.attend(q, codes, scales, np.arange(n), scale)
    V = dequant_ref(codes, scales)
    Z = scale * (bf16_ref(q) @ V.T)
    m = Z.max(axis=1, keepdims=True)
    P = np.exp(Z - m)
    ref = (P @ V) / P.sum(axis=1, keepdims=True)
    ref_lse = m[:, 0] + np.log(P.sum(axis=1))
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(out - ref) <= 1e-6 * rms)
    assert np.allclose(lse, ref_lse, rtol=1e-6, atol=1e-6)


def test_single_row_and_zero_query():
    D = 64
    codes, scales = small_cache(30, D, seed=4)
    V = dequant_ref(codes, scales)
    q = W.random_bf16_bits((2, D), 5, 12).numpy().view(np.uint16)
    out, lse = oracle.attend(q, codes, scales, np.array([-1, 7, -1]), 0.3)
    assert np.array_equal(out, np.broadcast_to(V[7].astype(np.float32), out.shape))
    assert np.allclose(lse, 0.3 * (bf16_ref(q) @ V[7]), rtol=1e-6)
    # q = 0: uniform weights, out = mean of the selected rows, lse = log K
    sel = np.array([3, 9, 9, 20])
    out0, lse0 = oracle.attend(np.zeros((1, D), np.uint16), codes, scales, sel, 1.0)
    assert np.allclose(out0[0], V[sel].mean(axis=0), rtol=1e-6, atol=1e-7)
    assert np.isclose(lse0[0], np.log(4.0))


def test_permutation_and_padding_invariance():
    D = 64
    codes, scales = small_cache(50, D, seed=6)
    q = W.random_bf16_bits((4, D), 7, 13).numpy().view(np.uint16)
    idx = np.array([4, 8, 15, 16, 23, 42])
    a, la = oracle.attend(q, codes, scales, idx, 0.125)
    b, lb = oracle.attend(q, codes, scales, np.concatenate([idx[::-1], [-1, -1]]), 0.125)
    assert np.allclose(a, b, rtol=1e-6, atol=1e-7) and np.allclose(la, lb, rtol=1e-7)


def test_empty_selection():
    codes, scales = small_cache(5, 32, seed=8)
    out, lse = oracle.attend(np.zeros((2, 32), np.uint16) + 0x3F80, codes, scales, np.array([-1, -1]), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------------------
# Mode invariants ("G2C Brief", section "CSA2: most layers don't keep their own cache")
# ---------------------------------------------------------------------------

def tiny_workload(**kw):
    base = dict(name="t", B=2, L=300, H=4, D=64, HI=3, DI=64, K=20)
    base.update(kw)
    return W.Workload(**base)


def build_cache(wl, seed=0):
    c = oracle.Cache(wl.B, wl.capacity, wl.D, wl.DI)
    lat = np.stack([W.cache_rows(wl, seed, b)[0].numpy() for b in range(wl.B)])
    ik = np.stack([W.cache_rows(wl, seed, b)[1].numpy() for b in range(wl.B)])
    c.append(lat, ik)
    return c


def test_reuse_of_full_indices_reproduces_full():
    wl = tiny_workload()
    cache = build_cache(wl)
    inp = W.layer_inputs(wl, 0, 0)
    full = oracle.run_layer(cache, oracle.FULL, inp, wl.K, wl.scale)
    prev = {u: r["idx"] for u, r in full.items()}
    reuse = oracle.run_layer(cache, oracle.REUSE, inp, wl.K, wl.scale, prev_idx=prev)
    for u in full:
        assert np.array_equal(full[u]["out"], reuse[u]["out"])
        assert np.array_equal(full[u]["lse"], reuse[u]["lse"])


def test_reindex_with_full_query_reproduces_full_selection():
    wl = tiny_workload()
    cache = build_cache(wl)
    inp = W.layer_inputs(wl, 0, 0)
    full = oracle.run_layer(cache, oracle.FULL, inp, wl.K, wl.scale, pool_keep=64)
    rx = oracle.run_layer(cache, oracle.REINDEX, inp, wl.K, wl.scale)
    # a pool that holds every block also reproduces the Full selection
    pool_all = {u: np.arange((wl.L + 7) // 8) for u in full}
    rxp = oracle.run_layer(cache, oracle.REINDEX, inp, wl.K, wl.scale, pool_in=pool_all)
    for u in full:
        assert np.array_equal(full[u]["idx"], rx[u]["idx"])
        assert np.array_equal(full[u]["idx"], rxp[u]["idx"])


def test_planted_block_reaches_pool_and_selection():
    wl = tiny_workload(B=1, L=2000, planted=16, pool_blocks=16, layers=(0, 1, 1), K=32, HI=4, DI=64)
    cache = build_cache(wl, seed=3)
    off = W.planted_offset(wl, 3)
    inputs = [W.layer_inputs(wl, 3, li) for li in range(3)]
    res = oracle.run_chain(cache, wl.layers, inputs, wl.K, wl.scale, pool_keep=wl.pool_blocks)
    planted_blocks = set(range(off // 8, (off + wl.planted - 1) // 8 + 1))
    pool = res[0][(0, 0)]["pool"]
    assert planted_blocks <= set(pool.tolist())
    for r in res:
        assert set(range(off, off + wl.planted)) <= set(r[(0, 0)]["idx"].tolist())


def test_causal_positions_and_append():
    """P positions after an append: position p sees length - P + 1 + p rows."""
    wl = tiny_workload(B=1, L=100, P=3, n_append=3, K=200)
    cache = build_cache(wl)
    app = W.append_rows(wl, 0)
    cache.append(app["rows"].numpy(), app["ikeys"].numpy())
    inp = W.layer_inputs(wl, 0, 0)
    res = oracle.run_layer(cache, oracle.FULL, inp, wl.K, wl.scale, P=3)
    for p in range(3):
        idx = res[(0, p)]["idx"]
        assert (idx >= 0).sum() == 101 + p           # K exceeds the visible rows
        assert idx.max() == 100 + p
