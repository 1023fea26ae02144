"""a3 on the GPU: top-K and the block pool on identical fp32 scores must equal
the oracle's selection exactly (same scores in, same sets out)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import ascending_then_padding, need_gpu

pytestmark = pytest.mark.gpu


def lengths_cache(Bn, cap, lengths):
    c = B.Cache(Bn, cap, 128, 64)
    c.lengths.copy_(torch.tensor(lengths, dtype=torch.int32))
    return c


def scores_with_ties(shape, seed, kind):
    s = W.random_scores(shape, seed).numpy()
    if kind == "ties":
        s = np.round(s * 4) / 4                 # many exact ties
    elif kind == "zeros":
        s = np.maximum(s, 0)                    # half exact zeros (the ReLU case)
        s[..., ::7] = -0.0
    elif kind == "negative":
        s = -np.abs(s) - 1
    return np.ascontiguousarray(s.astype(np.float32))


@pytest.mark.parametrize("n,K,kind", [(100, 256, "plain"), (256, 256, "plain"), (4096, 256, "plain"),
                                      (4096, 256, "ties"), (5000, 2048, "zeros"), (65536, 2048, "plain"),
                                      (65536, 2048, "ties"), (131072, 2048, "zeros"), (3, 1, "negative"),
                                      (1048576, 2048, "plain")])
def test_topk_equals_oracle(n, K, kind):
    need_gpu()
    Bn = 2 if n < 200000 else 1
    cap = (n + 3) // 4 * 4
    s = scores_with_ties((Bn, 1, cap), n + K, kind)
    cache = lengths_cache(Bn, cap, [n] * Bn)
    idx, _ = B.csa_topk(cache, torch.from_numpy(s).cuda(), K)
    got = idx.cpu().numpy()
    for b in range(Bn):
        ref = oracle.topk(s[b, 0, :n], K)
        assert sorted(got[b, 0][got[b, 0] >= 0].tolist()) == sorted(ref[ref >= 0].tolist())
        ascending_then_padding(got[b, 0])


def test_causal_positions_and_pool():
    need_gpu()
    P, cap = 6, 4000
    lengths = [3990, 17]
    s = scores_with_ties((2, P, cap), 5, "ties")
    cache = lengths_cache(2, cap, lengths)
    idx, pool = B.csa_topk(cache, torch.from_numpy(s).cuda(), 64, pool_keep=100)
    gi, gp = idx.cpu().numpy(), pool.cpu().numpy()
    for b in range(2):
        for p in range(P):
            L = max(lengths[b] - P + 1 + p, 0)
            ref = oracle.topk(s[b, p, :L], 64)
            assert sorted(gi[b, p][gi[b, p] >= 0].tolist()) == sorted(ref[ref >= 0].tolist())
            refp = oracle.build_pool(s[b, p, :L], 100) if L else -np.ones(100, np.int64)
            assert gp[b, p].tolist() == refp.tolist()


def test_select_over_pool_candidates():
    need_gpu()
    L, nblk = 5003, 300
    nb = (L + 7) // 8
    pool = np.full((1, 2, nblk), -1, np.int32)
    pool[0, 0] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=3).numpy().argsort()[:nblk])
    pool[0, 1, :50] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=4).numpy().argsort()[:49].tolist() + [nb - 1])
    s = scores_with_ties((1, 2, nblk * 8), 9, "ties")
    cache = lengths_cache(1, L + 1, [L + 1])           # P=2: position 0 sees L rows, position 1 sees L+1
    idx, _ = B.csa_topk(cache, torch.from_numpy(s).cuda(), 128, pool=torch.from_numpy(pool).cuda())
    gi = idx.cpu().numpy()
    for p in range(2):
        rows, valid = oracle.pool_rows(pool[0, p], L + p)
        sel = oracle.topk(s[0, p], 128, valid)
        ref = rows[sel[sel >= 0]]
        assert sorted(gi[0, p][gi[0, p] >= 0].tolist()) == sorted(ref.tolist())
        ascending_then_padding(gi[0, p])


def shaped_scores(n, kind, seed):
    """Score rows that drive each branch of the one-CTA selection: a few huge
    scores that stretch the key range so that the threshold bin of the first
    pass holds thousands of keys (another pass over all keys), a narrow band of
    distinct scores (several passes over the gathered list), and a band of
    exact ties at the K-th value (the tie rule); rows whose K-th largest score
    equals the selection's lower bound (the least of the largest of each run of
    8), and rows with exact zeros."""
    rng = np.random.default_rng(seed)
    if kind == "stretched":
        s = (1.0 + rng.random(n) * 1e-3).astype(np.float32)
        s[rng.choice(n, 384, replace=False)] = 1e30
    elif kind == "band":
        # 384 huge scores; 600 scores on 256 consecutive floats above 1 (two or
        # three copies each: the gathered list needs two passes, the second
        # down to single values); the rest near 0.5
        s = (0.5 + rng.random(n) * 1e-3).astype(np.float32)
        pick = rng.choice(n, 984, replace=False)
        s[pick[:384]] = 1e30
        s[pick[384:]] = np.float32(1.0) + (np.arange(600) % 256).astype(np.float32) * np.float32(2.0 ** -23)
    elif kind in ("group_max", "group_max_ties"):
        # every run of 8 candidates has its largest score 3.0 (the selection's
        # lower bound is then the K-th largest itself at K = n / 8); with
        # "group_max_ties" 100 more candidates tie at 3.0
        s = rng.random(n).astype(np.float32)
        s[np.arange(0, n - 7, 8) + rng.integers(0, 8, size=n // 8)] = 3.0
        if kind == "group_max_ties":
            s[rng.choice(np.flatnonzero(s < 3.0), 100, replace=False)] = 3.0
    elif kind == "relu_zeros":
        # 40 % exact zeros (every head's product negative), the rest positive
        s = rng.random(n).astype(np.float32) * 4.0
        s[rng.random(n) < 0.4] = 0.0
    else:  # "tie_cut": 1500 above, 1000 tied, the rest below
        s = rng.random(n).astype(np.float32)
        order = rng.permutation(n)
        s[order[:1500]] += 10.0
        s[order[1500:2500]] = 5.0
    return s


@pytest.mark.parametrize("n,K,kind", [(16384, 2048, "plain"), (16385, 2048, "plain"), (16384, 16384, "plain"),
                                      (16384, 1, "plain"), (16384, 2048, "stretched"), (9000, 700, "band"),
                                      (16384, 2048, "tie_cut"), (4097, 3000, "tie_cut"),
                                      (16384, 2048, "group_max"), (16384, 2048, "group_max_ties"),
                                      (16384, 2048, "relu_zeros"), (16384, 8000, "relu_zeros"),
                                      (9000, 2048, "relu_zeros"), (16384, 1000, "group_max")])
def test_one_cta_select_branches(n, K, kind):
    """Rows of 8,193 to 16,384 candidates are selected by select_one_kernel,
    longer ones by a cluster, shorter ones by select_kernel in one CTA; all
    equal the oracle."""
    need_gpu()
    cap = (n + 3) // 4 * 4
    if kind == "plain":
        s = scores_with_ties((1, 1, cap), n, "plain")[0, 0]
    else:
        s = np.zeros(cap, np.float32)
        s[:n] = shaped_scores(n, kind, n + K)
    cache = lengths_cache(1, cap, [n])
    idx, _ = B.csa_topk(cache, torch.from_numpy(s.reshape(1, 1, cap)).cuda(), K)
    got = idx.cpu().numpy()[0, 0]
    ref = oracle.topk(s[:n], K)
    assert got[got >= 0].tolist() == sorted(ref[ref >= 0].tolist())
    assert (got >= 0).sum() == min(n, K)
    ascending_then_padding(got)


@pytest.mark.parametrize("P,cap,lengths,keep,kind", [
    (6, 4000, [3990, 17], 100, "ties"),          # causal positions, a sequence shorter than the pool
    (1, 1 << 20, [1 << 20, 1000003], 2048, "zeros"),   # 131,072 blocks: the cluster path
    (1, 100000, [100000, 99999], 2048, "plain"),  # 12,500 blocks: the one-CTA path
    (1, 1 << 21, [1 << 21], 2048, "plain"),       # 262,144 blocks: two stages through the workspace
])
def test_pool_from_block_maxima(P, cap, lengths, keep, kind):
    """csa_topk given block maxima (here the oracle's, from the same scores)
    keeps the same pool as the oracle's build_pool, and the same top K rows."""
    need_gpu()
    Bn = len(lengths)
    s = scores_with_ties((Bn, P, cap), cap + keep, kind)
    cache = lengths_cache(Bn, cap, lengths)
    bm = B.block_max_buffer(cache, P)
    bmh = np.full(tuple(bm.shape), np.nan, np.float32)
    for b in range(Bn):
        for p in range(P):
            L = max(lengths[b] - P + 1 + p, 0)
            bmh[b, p, :(L + 7) // 8] = oracle.block_max(s[b, p, :L])
    bm.copy_(torch.from_numpy(bmh))
    K = 64 if cap < 10000 else 2048
    ws = torch.empty(max(16, B.topk_workspace_size(cache, P, K, 0, keep)), dtype=torch.uint8, device="cuda")
    idx, pool = B.csa_topk(cache, torch.from_numpy(s).cuda(), K, pool_keep=keep, block_max=bm, workspace=ws)
    gi, gp = idx.cpu().numpy(), pool.cpu().numpy()
    for b in range(Bn):
        for p in range(P):
            L = max(lengths[b] - P + 1 + p, 0)
            refp = oracle.build_pool(s[b, p, :L], keep) if L else -np.ones(keep, np.int64)
            assert gp[b, p].tolist() == refp.tolist(), (b, p)
            ref = oracle.topk(s[b, p, :L], K)
            assert sorted(gi[b, p][gi[b, p] >= 0].tolist()) == sorted(ref[ref >= 0].tolist()), (b, p)
            ascending_then_padding(gi[b, p])
