"""The context split on one GPU: a sequence's rows in G slices, each with its
own cache, the G ranks' steps run in turn in one process (the exchange is a
concatenation), against the single-cache path and the oracle.

"G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
index, select": every entry is scored, the best K are kept, the query attends
to those.  The split's claims, each checked here:
- a slice's pair scores are the single cache's scores of the same rows (the
  index score of a row depends on that row alone), so the global top K of the
  slices' top Ks is the single cache's top K: equal sets, up to members whose
  score equals the K-th score exactly (either may be kept);
- the selection agrees with the oracle's top K (check_topk's tolerance);
- the merged attention is within 2e-3 x RMS of the oracle's over the same
  selected rows, its lse within 1e-5;
- csa_topk_pairs, csa_select_pairs (rows and blocks of 8), csa_ids_window and
  csa_lse_merge against plain definitions, exactly where no arithmetic is
  involved.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import context_split as CS
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import ascending_then_padding, check_attention, check_topk, device_cache, need_gpu

pytestmark = pytest.mark.gpu


def split_parts(wl: W.Workload, lat, ik, G: int):
    parts = []
    for g in range(G):
        lo, hi = CS.slice_rows(wl.L, G, g)
        assert hi > lo
        cache = B.Cache(wl.B, hi - lo, wl.D, wl.DI)
        B.csa_quantize_append(cache, lat[:, lo:hi].contiguous(), ik[:, lo:hi].contiguous())
        parts.append(CS.Part(cache, lo, hi - lo))
    return parts


def same_selection(split_idx, whole_idx, whole_scores, what):
    """Equal sets, except members whose score equals the K-th score exactly."""
    a = set(int(x) for x in split_idx if x >= 0)
    b = set(int(x) for x in whole_idx if x >= 0)
    assert len(a) == len(b), (what, len(a), len(b))
    if a == b:
        return
    kth = min(whole_scores[i] for i in b)
    diff = sorted(a ^ b)
    assert all(whole_scores[i] == kth for i in diff), (what, diff[:8], [whole_scores[i] for i in diff[:8]], kth)


CASES = [
    # name, G, workload, layers checked by the oracle's top K
    ("g2_ragged", 2, W.Workload("g2", B=2, L=40003, H=64, D=512, HI=64, DI=128, K=2048, outlier_channels=5,
                                layers=(W.FULL, W.REINDEX, W.REUSE, W.REINDEX)), True),
    ("g3_short_slices", 3, W.Workload("g3", B=2, L=5003, H=16, D=128, HI=16, DI=64, K=2048,
                                      layers=(W.FULL, W.REUSE, W.REINDEX)), True),
    ("g5_small_k", 5, W.Workload("g5", B=3, L=20000, H=8, D=256, HI=32, DI=128, K=7,
                                 layers=(W.FULL, W.REINDEX)), True),
    ("g8_1m", 8, W.Workload("g8", B=1, L=1 << 20, H=64, D=512, HI=64, DI=128, K=2048,
                            layers=(W.FULL, W.REUSE)), False),
]


@pytest.mark.parametrize("name,G,wl,oracle_topk", CASES, ids=[c[0] for c in CASES])
def test_split_chain(name, G, wl, oracle_topk):
    need_gpu()
    seed = 29
    whole, lat, ik = device_cache(wl, seed)
    parts = split_parts(wl, lat, ik, G)
    ikh = ik.cpu().numpy() if oracle_topk else None
    prev = None
    for li, mode in enumerate(wl.layers):
        inp = W.layer_inputs(wl, seed, li, device="cuda")
        if mode != W.REUSE:
            pairs = [CS.local_pairs(p, inp["iq"], inp["w"], wl.K) for p in parts]
            prev = CS.global_selection([s for s, _ in pairs], [i for _, i in pairs], wl.K)
            scores = B.csa_index_score(whole, inp["iq"], inp["w"])
            idx_whole, _ = B.csa_topk(whole, scores, wl.K)
            torch.cuda.synchronize()
            s = scores.cpu().numpy()
            # each pair's score is the single cache's score of its row, bit for bit
            for (ps, pi) in pairs:
                ps, pi = ps.cpu().numpy(), pi.cpu().numpy()
                for b in range(wl.B):
                    v = pi[b, 0] >= 0
                    assert np.array_equal(ps[b, 0][v], s[b, 0][pi[b, 0][v]]), (name, li, b)
                    assert np.all(np.isneginf(ps[b, 0][~v]))
            gi, wi = prev.cpu().numpy(), idx_whole.cpu().numpy()
            for b in range(wl.B):
                ascending_then_padding(gi[b, 0])
                assert (gi[b, 0] >= 0).sum() == min(wl.K, wl.L)
                same_selection(gi[b, 0], wi[b, 0], s[b, 0], (name, li, b))
                if oracle_topk:
                    rows = np.arange(wl.L, dtype=np.int64)
                    sc = oracle.index_scores(inp["iq"][b, 0].cpu().numpy(), inp["w"][b, 0].cpu().numpy(),
                                             ikh[b], rows, threads=8)
                    want = oracle.topk(sc, wl.K)
                    check_topk(gi[b, 0], want, lambda r: sc[r], wl.K, (name, li, b))
        partial = [CS.local_attention(p, inp["q"], prev, wl.scale) for p in parts]
        out, lse = CS.merge([o for o, _ in partial], [l for _, l in partial])
        torch.cuda.synchronize()
        assert B.csa_device_status() == 0
        o, l, gi, qh = out.cpu().numpy(), lse.cpu().numpy(), prev.cpu().numpy(), inp["q"].cpu().numpy()
        for b in range(wl.B):
            # the oracle quantises the selected rows itself (row by row, as the cache does)
            sel = gi[b, 0][gi[b, 0] >= 0].astype(np.int64)
            codes, scales = oracle.quantize_rows(lat[b, torch.tensor(sel, device="cuda")].cpu().numpy()[None])
            ro, rl = oracle.attend(qh[b, 0], codes[0], scales[0], np.arange(sel.shape[0]), wl.scale)
            check_attention(o[b, 0], ro, (name, li, b))
            assert np.allclose(l[b, 0], rl, rtol=1e-5, atol=1e-5), (name, li, b)


@pytest.mark.parametrize("rows,n,K,levels", [(4, 2 * 2048, 2048, 0), (3, 8 * 2048, 2048, 64), (2, 1000, 1500, 5),
                                             (5, 3 * 7, 7, 3), (1, 262144, 16384, 0)])
def test_topk_pairs_exact(rows, n, K, levels):
    """The K best pairs (ties: the earlier pair; id -1 = empty) in pair order,
    equal to the oracle's top K of the same fp32 values."""
    need_gpu()
    rng = np.random.default_rng(rows * 1000 + K)
    ps = rng.standard_normal((rows, n)).astype(np.float32)
    if levels:  # few distinct values: many exact ties
        ps = np.round(ps * levels / 4).astype(np.float32)
    pi = np.sort(rng.choice(1 << 30, size=(rows, n), replace=False), axis=-1).astype(np.int32)
    empty = rng.random((rows, n)) < 0.1
    pi[empty] = -1
    ps[empty] = -np.inf
    got = B.csa_topk_pairs(torch.tensor(ps, device="cuda"), torch.tensor(pi, device="cuda"), K).cpu().numpy()
    for r in range(rows):
        sel = oracle.topk(ps[r], K, (pi[r] >= 0).astype(np.uint8))
        sel = np.sort(sel[sel >= 0])
        want = np.full(K, -1, np.int32)
        want[:sel.shape[0]] = pi[r, sel]
        assert np.array_equal(got[r], want), (r, np.flatnonzero(got[r] != want)[:8])


@pytest.mark.parametrize("block", [1, 8])
def test_select_pairs(block):
    need_gpu()
    rng = np.random.default_rng(block)
    Bn, cap, n = 3, 4099, 300
    cache = B.Cache(Bn, cap, 128, 64)
    lengths = np.array([4099, 4001, 17], np.int32)
    cache.lengths.copy_(torch.tensor(lengths))
    ld = (cap + 3) // 4 * 4
    s = rng.standard_normal((Bn, 1, ld)).astype(np.float32)
    ids_max = (cap + block - 1) // block
    idx = rng.integers(-1, ids_max, size=(Bn, 1, n)).astype(np.int32)
    ps, pi = B.csa_select_pairs(cache, torch.tensor(s, device="cuda"), torch.tensor(idx, device="cuda"), block, 1234)
    ps, pi = ps.cpu().numpy(), pi.cpu().numpy()
    for b in range(Bn):
        for j in range(n):
            i = int(idx[b, 0, j])
            if i < 0:
                assert pi[b, 0, j] == -1 and np.isneginf(ps[b, 0, j])
                continue
            assert pi[b, 0, j] == i + 1234
            r = np.arange(i * block, i * block + block)
            r = r[r < lengths[b]]
            want = s[b, 0, r].max() if r.size else -np.inf
            assert ps[b, 0, j] == want, (b, j)


def test_ids_window():
    need_gpu()
    rng = np.random.default_rng(3)
    ids = rng.integers(-1, 100000, size=(7, 1, 2048)).astype(np.int32)
    got = B.csa_ids_window(torch.tensor(ids, device="cuda"), 30000, 61000).cpu().numpy()
    want = np.where((ids >= 30000) & (ids < 61000), ids - 30000, -1)
    assert np.array_equal(got, want)


def test_lse_merge():
    """Against the merge written out in double; a part with lse = -inf has no
    rows, a unit with no rows in any part gives out 0, lse -inf."""
    need_gpu()
    rng = np.random.default_rng(11)
    parts, units, H, D = 4, 6, 16, 512
    outs = rng.standard_normal((parts, units, H, D)).astype(np.float32)
    lses = (rng.standard_normal((parts, units, H)) * 20).astype(np.float32)
    lses[1, 2] = -np.inf
    lses[:, 4, 3] = -np.inf
    out, lse = B.csa_lse_merge(torch.tensor(outs, device="cuda"), torch.tensor(lses, device="cuda"))
    out, lse = out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    l = lses.astype(np.float64)
    for u in range(units):
        for h in range(H):
            v = np.isfinite(l[:, u, h])
            if not v.any():
                assert np.all(out[u, h] == 0) and np.isneginf(lse[u, h])
                continue
            m = l[v, u, h].max()
            wgt = np.exp(l[v, u, h] - m)
            want = (wgt[:, None] * outs[v, u, h].astype(np.float64)).sum(0) / wgt.sum()
            assert np.allclose(out[u, h], want, rtol=1e-5, atol=1e-6), (u, h)
            assert abs(lse[u, h] - (m + np.log(wgt.sum()))) <= 1e-5 * max(1.0, abs(m)), (u, h)
