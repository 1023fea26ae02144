"""Pins of the oracle's indexer score (a2/a4) and selection (a3, pool) on the CPU."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import workloads as W


def e4m3_to_f64(b):
    """Decode E4M3 bytes with torch's own cast (independent of the oracle)."""
    t = torch.as_tensor(np.ascontiguousarray(b)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def draw(HI, DI, n, seed):
    iq = W.random_e4m3_bytes((HI, DI), seed, 1).numpy()
    ik = W.random_e4m3_bytes((n, DI), seed, 2).numpy()
    w = W.random_uniform((HI,), seed, 3).numpy().astype(np.float32)
    return iq, ik, w


def test_single_head_unit_weight_is_relu_dot():
    """HI=1, w=1: score = ReLU(q . k), a plain library dot product."""
    iq, ik, _ = draw(1, 64, 300, seed=5)
    got = oracle.index_scores(iq, np.ones(1, np.float32), ik, np.arange(300))
    ref = np.maximum(e4m3_to_f64(ik) @ e4m3_to_f64(iq)[0], 0.0).astype(np.float32)
    assert np.array_equal(got, ref)
    assert (got == 0).sum() > 50              # the ReLU branch is exercised


def test_relu_identity_recovers_linear_form():
    """ReLU(x) - ReLU(-x) = x, so score(iq) - score(-iq) = sum_h w_h q_h.k, a
    library matrix product; catches sign, head and index errors."""
    iq, ik, w = draw(8, 128, 257, seed=6)
    rows = np.arange(257)
    pos = oracle.index_scores(iq, w, ik, rows).astype(np.float64)
    neg = oracle.index_scores(iq ^ np.uint8(0x80), w, ik, rows).astype(np.float64)
    lin = (e4m3_to_f64(ik) @ e4m3_to_f64(iq).T) @ w.astype(np.float64)
    scale = np.abs(pos) + np.abs(neg) + 1.0
    assert np.all(np.abs((pos - neg) - lin) <= 2e-7 * scale)


def test_head_permutation_and_weight_scaling():
    iq, ik, w = draw(6, 64, 100, seed=7)
    rows = np.arange(100)
    base = oracle.index_scores(iq, w, ik, rows)
    perm = np.array([3, 0, 5, 1, 4, 2])
    assert np.array_equal(oracle.index_scores(iq[perm], w[perm], ik, rows), base) or \
        np.allclose(oracle.index_scores(iq[perm], w[perm], ik, rows), base, rtol=1e-7, atol=0)
    assert np.array_equal(oracle.index_scores(iq, 2 * w, ik, rows), 2 * base)
    w0 = w.copy(); w0[2] = 0
    only2 = oracle.index_scores(iq[2:3], np.ones(1, np.float32), ik, rows).astype(np.float64)
    diff = base.astype(np.float64) - oracle.index_scores(iq, w0, ik, rows).astype(np.float64)
    assert np.allclose(diff, w[2] * only2, rtol=1e-6, atol=1e-5)


def test_row_gather_matches_full_scan():
    iq, ik, w = draw(4, 64, 200, seed=8)
    full = oracle.index_scores(iq, w, ik, np.arange(200))
    rows = np.array([199, 0, 17, 17, 64])
    assert np.array_equal(oracle.index_scores(iq, w, ik, rows), full[rows])


@pytest.mark.parametrize("trial", range(40))
def test_topk_brute_force_tiny_with_ties(trial):
    n = 1 + trial % 23
    K = 1 + (trial * 7) % 30
    vals = W.random_ints((n,), 0, 4, seed=100 + trial).numpy().astype(np.float32)
    vals[vals == 3] = -0.0                    # -0 ties with +0
    vals[vals == 2] = 0.0
    got = oracle.topk(vals, K)
    ref = sorted(range(n), key=lambda i: (-float(vals[i]), i))[:K]
    ref = ref + [-1] * (K - len(ref))
    assert got.tolist() == ref


def test_topk_validity_mask():
    s = W.random_scores((50,), seed=3).numpy()
    valid = (np.arange(50) % 3 != 0).astype(np.uint8)
    got = oracle.topk(s, 60, valid)
    keep = [i for i in range(50) if valid[i]]
    ref = sorted(keep, key=lambda i: (-float(s[i]), i))
    assert got.tolist() == ref + [-1] * (60 - len(ref))


@pytest.mark.parametrize("n,keep", [(64, 3), (61, 4), (8, 5), (1000, 20), (4097, 2048)])
def test_pool_is_best_blocks(n, keep):
    """Every kept block's best member beats (or ties at a higher id) every
    dropped block's; the partial last block uses only the rows it has."""
    s = W.random_scores((n,), seed=n).numpy()
    s[5] = s.max() + 1.0
    pool = oracle.build_pool(s, keep)
    nb = (n + 7) // 8
    padded = np.full(nb * 8, -np.inf, np.float32)
    padded[:n] = s
    bmax = padded.reshape(nb, 8).max(axis=1)
    kept = pool[pool >= 0]
    assert np.all(np.diff(kept) > 0)                         # ascending, unique
    assert kept.size == min(keep, nb)
    assert 0 in kept                                         # block of row 5
    dropped = np.setdiff1d(np.arange(nb), kept)
    if dropped.size:
        worst_kept = min((bmax[j], -j) for j in kept)
        best_dropped = max((bmax[j], -j) for j in dropped)
        assert worst_kept > best_dropped
    assert np.all(pool[kept.size:] == -1)


def test_pool_rows_layout():
    rows, valid = oracle.pool_rows([0, 2, -1], L_p=21)
    assert rows[:8].tolist() == list(range(8))
    assert rows[8:16].tolist() == list(range(16, 21)) + [0, 0, 0]
    assert valid.tolist() == [1] * 8 + [1] * 5 + [0] * 3 + [0] * 8
