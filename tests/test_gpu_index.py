"""a2/a4 on the GPU: indexer scores against the oracle (full scan, pool rows,
several causal positions)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import device_cache, need_gpu

pytestmark = pytest.mark.gpu


def e4m3_f64(b):
    return torch.as_tensor(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def abs_bound(iq, w, ik_rows):
    """sum_h w_h sum_d |q_hd k_d|: the scale of an fp32 rounding error bound."""
    return np.abs(e4m3_f64(ik_rows)) @ np.abs(e4m3_f64(iq)).T @ np.abs(w.astype(np.float64))


def compare(gpu, ora, bound, what):
    err = np.abs(gpu.astype(np.float64) - ora.astype(np.float64))
    tol = 1e-5 * bound + 1e-30
    assert np.all(err <= tol), (what, float((err / np.maximum(bound, 1e-30)).max()))


@pytest.mark.parametrize("HI,DI,P", [(4, 64, 1), (64, 128, 1), (16, 128, 3), (64, 64, 6)])
def test_full_scan_scores(HI, DI, P):
    need_gpu()
    wl = W.Workload("t", B=2, L=3001, H=4, D=128, HI=HI, DI=DI, K=8, P=P)
    cache, _, ik = device_cache(wl, seed=11)
    inp = W.layer_inputs(wl, 11, 0, device="cuda")
    scores = B.csa_index_score(cache, inp["iq"], inp["w"])
    torch.cuda.synchronize()
    s = scores.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        for p in range(P):
            L = wl.L - P + 1 + p
            ora = oracle.index_scores(iqh[b, p], wh[b, p], ikh[b], np.arange(L))
            compare(s[b, p, :L], ora, abs_bound(iqh[b, p], wh[b, p], ikh[b, :L]), (b, p))


def test_pool_scores_with_ragged_tail():
    need_gpu()
    wl = W.Workload("t", B=2, L=2003, H=4, D=128, HI=16, DI=128, K=8)
    cache, _, ik = device_cache(wl, seed=12)
    inp = W.layer_inputs(wl, 12, 0, device="cuda")
    nb = (wl.L + 7) // 8
    pool = np.full((wl.B, 1, 40), -1, np.int32)
    pool[0, 0, :37] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=1).numpy().argsort()[:37])
    pool[1, 0, :40] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=2).numpy().argsort()[:39].tolist() + [nb - 1])
    scores = B.csa_index_score(cache, inp["iq"], inp["w"], pool=torch.from_numpy(pool).cuda())
    torch.cuda.synchronize()
    s = scores.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        rows, valid = oracle.pool_rows(pool[b, 0], wl.L)
        ora = oracle.index_scores(iqh[b, 0], wh[b, 0], ikh[b], rows)
        v = valid.astype(bool)
        compare(s[b, 0, :320][v], ora[v], abs_bound(iqh[b, 0], wh[b, 0], ikh[b, rows[v]]), b)


@pytest.mark.parametrize("L,P", [(3001, 3), (4096, 1), (17, 2)])
def test_block_maxima(L, P):
    """The scan's block maxima ("G2C Brief", "The hierarchical indexer": a block
    of 8 rows is ranked by its best member): each block's entry equals the
    largest of the same call's row scores below L_p bit for bit, and the
    oracle's block maximum within the scores' bound; the row scores are those
    of the call without block maxima."""
    need_gpu()
    wl = W.Workload("t", B=2, L=L, H=4, D=128, HI=16, DI=128, K=8, P=P)
    cache, _, ik = device_cache(wl, seed=13)
    inp = W.layer_inputs(wl, 13, 0, device="cuda")
    bm = B.block_max_buffer(cache, P)
    bm.fill_(float("nan"))
    scores = B.csa_index_score(cache, inp["iq"], inp["w"], block_max=bm)
    plain = B.csa_index_score(cache, inp["iq"], inp["w"])
    torch.cuda.synchronize()
    s, g, s0 = scores.cpu().numpy(), bm.cpu().numpy(), plain.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        for p in range(P):
            Lp = wl.L - P + 1 + p
            nb = (Lp + 7) // 8
            assert np.array_equal(s[b, p, :Lp], s0[b, p, :Lp]), (b, p)
            assert np.array_equal(g[b, p, :nb], oracle.block_max(s[b, p, :Lp])), (b, p)
            ora = oracle.index_scores(iqh[b, p], wh[b, p], ikh[b], np.arange(Lp))
            bound = abs_bound(iqh[b, p], wh[b, p], ikh[b, :Lp])
            bb = np.zeros(nb * 8)
            bb[:Lp] = bound
            compare(g[b, p, :nb], oracle.block_max(ora.astype(np.float32)), bb.reshape(nb, 8).max(1), (b, p))
