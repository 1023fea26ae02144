"""a4 on the GPU: a Reindex layer over the hierarchical pool in one call
(csa_pool_topk, in both forms: one cluster that selects on chip, and one CTA
per 128 rows whose last CTA selects, the form csa_layer_step takes), against
the oracle's scoring of the pool's rows and its top-K.

The GPU scores in fp32 and the oracle in double, so the selected sets must be
equal except for members whose oracle score is within 1e-5 relative of the
oracle's K-th score (check_topk).  Cases: pools of 128, 300 (ragged cluster
shares) and 2,048 blocks; -1 padding and out-of-range block ids; causal
positions whose visible length cuts pool blocks; K above the number of valid
rows; 16, 32, 48 (padded to 64) and 64 indexer heads; 64- and 128-byte keys;
duplicated key rows, whose scores tie exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import ascending_then_padding, check_topk, need_gpu

pytestmark = pytest.mark.gpu


def make_pool(rng, P, nblk, cap_blocks, n_valid):
    """Ascending block ids, -1 padded, per position."""
    pool = np.full((P, nblk), -1, np.int64)
    for p in range(P):
        ids = np.sort(rng.choice(cap_blocks, size=n_valid, replace=False))
        pool[p, :n_valid] = ids
    return pool


@pytest.mark.parametrize("form", ["cluster", "spread"])
@pytest.mark.parametrize("HI,DI,nblk,n_valid,K,P,L", [
    (64, 128, 2048, 2048, 2048, 1, 1048576 // 16),
    (64, 128, 2048, 1900, 2048, 2, 40000),
    (32, 128, 300, 290, 700, 2, 20000),
    (16, 64, 128, 128, 256, 1, 5000),
    (48, 128, 512, 500, 4000, 3, 9000),
    (64, 64, 1000, 1000, 1, 1, 30000),
])
def test_pool_topk_matches_oracle(HI, DI, nblk, n_valid, K, P, L, form):
    need_gpu()
    seed = 61
    rng = np.random.default_rng(seed)
    wl = W.Workload("pool", B=2, L=L, H=16, D=128, HI=HI, DI=DI, K=K, P=P)
    cache = B.Cache(wl.B, wl.capacity, wl.D, wl.DI)
    lat = torch.zeros((wl.B, wl.L, wl.D), dtype=torch.int16, device="cuda")
    ik = torch.empty((wl.B, wl.L, wl.DI), dtype=torch.uint8, device="cuda")
    for b in range(wl.B):
        _, ik[b] = W.cache_rows(wl, seed, b, device="cuda")
    # duplicated key rows: exact score ties
    ik[:, 100:140] = ik[:, 200:240]
    B.csa_quantize_append(cache, lat, ik)
    inp = W.layer_inputs(wl, seed, 1, device="cuda")
    cap_blocks = (wl.capacity + 7) // 8
    pool = np.stack([make_pool(rng, P, nblk, cap_blocks, n_valid) for _ in range(wl.B)])
    pool[0, 0, 3] = -1 if n_valid > 3 else pool[0, 0, 3]      # a hole inside the pool
    pool_t = torch.tensor(pool, dtype=torch.int32, device="cuda")
    ws = None
    if form == "spread":
        ws = torch.empty(B.pool_topk_workspace_size(cache, P, nblk), dtype=torch.uint8, device="cuda")
    idx = B.csa_pool_topk(cache, inp["iq"], inp["w"], pool_t, K, workspace=ws)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    gi = idx.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        for p in range(P):
            Lp = oracle.visible_length(wl.L, P, p)
            rows, valid = oracle.pool_rows(pool[b, p], Lp)
            sc = oracle.index_scores(iqh[b, p], wh[b, p], ikh[b], rows)
            sel = oracle.topk(sc, K, valid)
            want = np.where(sel >= 0, rows[np.maximum(sel, 0)], -1)
            by_row = dict(zip(rows[valid > 0].tolist(), sc[valid > 0].tolist()))
            ascending_then_padding(gi[b, p])
            check_topk(gi[b, p], want, lambda r: np.array([by_row[int(x)] for x in r], np.float32), K, (b, p))
            assert (gi[b, p] >= 0).sum() == min(K, int(valid.sum()))


def test_pool_topk_agrees_with_two_calls():
    """Both forms of the fused call and csa_index_score + csa_topk over the
    same pool select the same rows (their fp32 scores differ only in summation
    order); the two fused forms score identically, so they select identically,
    and calling the spread form again (its counters back at 0) repeats it."""
    need_gpu()
    wl = W.Workload("pool2", B=1, L=100000, H=16, D=128, HI=64, DI=128, K=2048)
    cache = B.Cache(wl.B, wl.capacity, wl.D, wl.DI)
    lat = torch.zeros((wl.B, wl.L, wl.D), dtype=torch.int16, device="cuda")
    _, ik = W.cache_rows(wl, 7, 0, device="cuda")
    B.csa_quantize_append(cache, lat, ik[None].contiguous())
    inp = W.layer_inputs(wl, 7, 1, device="cuda")
    rng = np.random.default_rng(7)
    pool = torch.tensor(make_pool(rng, 1, 2048, (wl.L + 7) // 8, 2048)[None], dtype=torch.int32, device="cuda")
    fused = B.csa_pool_topk(cache, inp["iq"], inp["w"], pool, wl.K)
    ws = torch.empty(B.pool_topk_workspace_size(cache, 1, 2048), dtype=torch.uint8, device="cuda")
    spread = [B.csa_pool_topk(cache, inp["iq"], inp["w"], pool, wl.K, workspace=ws) for _ in range(3)]
    scores = B.csa_index_score(cache, inp["iq"], inp["w"], pool=pool)
    two, _ = B.csa_topk(cache, scores, wl.K, pool=pool)
    torch.cuda.synchronize()
    s = scores[0, 0].cpu().numpy()
    rows = (pool[0, 0].cpu().numpy()[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    by_row = dict(zip(rows.tolist(), s.tolist()))
    check_topk(fused[0, 0].cpu().numpy(), two[0, 0].cpu().numpy(),
               lambda r: np.array([by_row[int(x)] for x in r], np.float32), wl.K)
    for sp in spread:
        assert torch.equal(sp, fused)
    assert B.csa_device_status() == 0
