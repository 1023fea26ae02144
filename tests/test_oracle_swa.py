"""Pins of the oracle's joint attention over the selected global entries and
the local sliding window (the first "next" row).

"DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section "The
Paper": the selected entries are glued onto the sliding-window KV and the query
attends to both.  "G2C Brief - DeepSeek V4.1-Flash", section "Two attention
paths in every layer": the local branch is exact attention over the most
recent 128 tokens; section "FP4 cache entries, and why they're safe": the
local cache stays in FP8.

Every reference here decodes with torch's FP8 cast and a literal E2M1 table,
not with the oracle's decoders.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import workloads as W
from test_oracle_attend import bf16_ref, dequant_ref, small_cache


def e4m3_ref(rows):
    return torch.as_tensor(np.ascontiguousarray(rows)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dense(q_bits, vecs, scale):
    """Plain softmax attention of every head over the given vectors (K = V)."""
    q = bf16_ref(q_bits)
    z = scale * q @ vecs.T
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    return p @ vecs / l, (m + np.log(l))[:, 0]


def setup(D=64, H=5, n=50, n_swa=140, seed=0):
    codes, scales = small_cache(n, D, seed=seed + 1)
    swa = W.random_e4m3_bytes((n_swa, D), seed + 2).numpy()
    q = W.random_bf16_bits((H, D), seed + 3).numpy().view(np.uint16)
    return codes, scales, swa, q, 1.0 / np.sqrt(D)


def test_window_only_equals_dense_attention_over_the_window():
    codes, scales, swa, q, scale = setup()
    idx = np.full(7, -1)
    out, lse = oracle.attend_swa(q, codes, scales, idx, swa, 12, 140, scale)
    ref, rl = dense(q, e4m3_ref(swa[12:140]), scale)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)
    assert np.allclose(lse, rl, rtol=1e-5, atol=1e-6)


def test_empty_window_equals_sparse_attention():
    codes, scales, swa, q, scale = setup()
    idx = np.array([3, -1, 40, 7, 7, 0])
    out, lse = oracle.attend_swa(q, codes, scales, idx, swa, 30, 30, scale)
    o2, l2 = oracle.attend(q, codes, scales, idx, scale)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_joint_softmax_is_dense_attention_over_the_union():
    codes, scales, swa, q, scale = setup(D=128, H=16, n=300, n_swa=200, seed=5)
    idx = np.array([5, 299, -1, 17, 150, 17, 0])
    out, lse = oracle.attend_swa(q, codes, scales, idx, swa, 72, 200, scale)
    sel = dequant_ref(codes[idx[idx >= 0]], scales[idx[idx >= 0]])
    vecs = np.concatenate([sel, e4m3_ref(swa[72:200])], axis=0)
    ref, rl = dense(q, vecs, scale)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)
    assert np.allclose(lse, rl, rtol=1e-5, atol=1e-6)


def test_log_sum_exp_merge_of_the_two_branches():
    """The joint result is the log-sum-exp merge of the two branches computed
    apart (the decomposition a split kernel relies on)."""
    codes, scales, swa, q, scale = setup(seed=9)
    idx = np.array([1, 2, 30, -1, 44])
    o1, l1 = oracle.attend(q, codes, scales, idx, scale)
    o2, l2 = oracle.attend_swa(q, codes, scales, np.full(1, -1), swa, 0, 128, scale)
    oj, lj = oracle.attend_swa(q, codes, scales, idx, swa, 0, 128, scale)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    assert np.allclose(oj, merged, rtol=1e-5, atol=1e-6)
    assert np.allclose(lj, m + np.log(w1 + w2), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("n_swa,P,W,want", [(200, 1, 128, [(72, 200)]), (130, 3, 128, [(0, 128), (1, 129), (2, 130)]),
                                            (5, 2, 128, [(0, 4), (0, 5)]), (300, 6, 4, [(291, 295), (292, 296), (293, 297), (294, 298), (295, 299), (296, 300)])])
def test_window_rows_of_each_position(n_swa, P, W, want):
    assert [oracle.swa_window(n_swa, P, p, W) for p in range(P)] == want
