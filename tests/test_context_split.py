"""The context split of one sequence over several ranks (row slices), host
logic on CPU with two gloo ranks.

Each rank holds a contiguous slice of every sequence's rows; a layer scores
the slice, keeps its local top K as (score, global id) pairs, gathers every
rank's pairs, takes the global top K, attends over its own selected rows and
merges every rank's partial output by log-sum-exp
(fp4_compressed_sparse_append_b300.context_split).  Here the device steps are
the oracle's (OracleOps, test code), so this test checks the split itself:
the slices, the id offsets, the two exchanges, the global selection and the
merge, against the oracle's chain over the whole sequence.  The library's
kernels for those steps are checked on a GPU in test_gpu_context_split.py.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from fp4_compressed_sparse_append_b300 import context_split as CS  # noqa: E402
from fp4_compressed_sparse_append_b300 import workloads as W  # noqa: E402

WL = W.Workload("split", B=2, L=3000, H=8, D=128, HI=4, DI=64, K=300,
                layers=(W.FULL, W.REINDEX, W.REUSE, W.REINDEX))
SEED = 5


class OracleOps:
    """The split's device steps computed by the oracle on host tensors
    ([B, 1, ...] shapes, as the library's calls take them)."""

    @staticmethod
    def index_score(cache, iq, w):
        ld = (cache.capacity + 3) // 4 * 4
        out = np.zeros((cache.B, 1, ld), np.float32)
        for b in range(cache.B):
            L = int(cache.lengths[b])
            out[b, 0, :L] = oracle.index_scores(iq[b, 0].numpy(), w[b, 0].numpy(), cache.ikeys[b],
                                                np.arange(L, dtype=np.int64))
        return torch.from_numpy(out)

    @staticmethod
    def topk(cache, scores, K):
        out = np.full((cache.B, 1, K), -1, np.int32)
        for b in range(cache.B):
            sel = oracle.topk(scores[b, 0, :int(cache.lengths[b])].numpy(), K)
            sel = np.sort(sel[sel >= 0])
            out[b, 0, :sel.shape[0]] = sel
        return torch.from_numpy(out)

    @staticmethod
    def select_pairs(cache, scores, idx, id_offset):
        s, i = scores.numpy(), idx.numpy()
        ps = np.where(i >= 0, np.take_along_axis(s, np.maximum(i, 0), axis=-1), -np.inf).astype(np.float32)
        pi = np.where(i >= 0, i + id_offset, -1).astype(np.int32)
        return torch.from_numpy(ps), torch.from_numpy(pi)

    @staticmethod
    def topk_pairs(pair_scores, pair_ids, K):
        ps, pi = pair_scores.numpy(), pair_ids.numpy()
        out = np.full((ps.shape[0], K), -1, np.int32)
        for r in range(ps.shape[0]):
            sel = oracle.topk(ps[r], K, (pi[r] >= 0).astype(np.uint8))
            sel = np.sort(sel[sel >= 0])              # pair order
            out[r, :sel.shape[0]] = pi[r, sel]
        return torch.from_numpy(out)

    @staticmethod
    def ids_window(ids, lo, hi):
        i = ids.numpy()
        return torch.from_numpy(np.where((i >= lo) & (i < hi), i - lo, -1).astype(np.int32))

    @staticmethod
    def attend(cache, q, idx, scale):
        H, D = q.shape[-2], q.shape[-1]
        out = np.zeros((cache.B, 1, H, D), np.float32)
        lse = np.zeros((cache.B, 1, H), np.float32)
        for b in range(cache.B):
            out[b, 0], lse[b, 0] = oracle.attend(q[b, 0].numpy(), cache.codes[b], cache.scales[b],
                                                 idx[b, 0].numpy().astype(np.int64), scale)
        return torch.from_numpy(out), torch.from_numpy(lse)

    @staticmethod
    def lse_merge(outs, lses):
        o, l = outs.numpy().astype(np.float64), lses.numpy().astype(np.float64)
        M = l.max(axis=0)
        safe = np.where(np.isfinite(M), M, 0.0)
        wgt = np.where(np.isfinite(l), np.exp(l - safe), 0.0)
        S = wgt.sum(axis=0)
        out = (wgt[..., None] * o).sum(axis=0) / np.where(S > 0, S, 1.0)[..., None]
        lse = np.where(S > 0, safe + np.log(np.where(S > 0, S, 1.0)), -np.inf)
        return torch.from_numpy(out.astype(np.float32)), torch.from_numpy(lse.astype(np.float32))


def _inputs():
    lat = torch.stack([W.cache_rows(WL, SEED, b, device="cpu")[0] for b in range(WL.B)])
    ik = torch.stack([W.cache_rows(WL, SEED, b, device="cpu")[1] for b in range(WL.B)])
    layers = [W.layer_inputs(WL, SEED, li, device="cpu") for li in range(len(WL.layers))]
    return lat, ik, layers


def run_split(rank, world, gather):
    """This rank's run of the chain; returns [(idx_global, out, lse)] per layer."""
    lat, ik, layers = _inputs()
    lo, hi = CS.slice_rows(WL.L, world, rank)
    cache = oracle.Cache(WL.B, hi - lo, WL.D, WL.DI)
    cache.append(lat[:, lo:hi].numpy(), ik[:, lo:hi].numpy())
    part = CS.Part(cache, lo, hi - lo)
    results, prev = [], None
    for li, mode in enumerate(WL.layers):
        inp = layers[li]
        if mode == W.REUSE:
            res = CS.layer_step(part, inp["q"], WL.K, WL.scale, gather, idx_global=prev, ops=OracleOps)
        else:
            res = CS.layer_step(part, inp["q"], WL.K, WL.scale, gather, iq=inp["iq"], w=inp["w"], ops=OracleOps)
            prev = res[0]
        results.append(tuple(t.numpy() for t in res))
    return results


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = run_split(rank, world, CS.torch_gather())
    dist.destroy_process_group()


def check_against_whole_sequence(results):
    """The split's selections equal the oracle's over the whole sequence exactly
    (the global top K of the ranks' top Ks is the top K), and its merged
    attention is within 2e-3 x RMS of the oracle's."""
    lat, ik, layers = _inputs()
    whole = oracle.Cache(WL.B, WL.L, WL.D, WL.DI)
    whole.append(lat.numpy(), ik.numpy())
    inputs = [{k: v.numpy() for k, v in inp.items()} for inp in layers]
    ref = oracle.run_chain(whole, WL.layers, inputs, WL.K, WL.scale, P=1)
    for li, (idx, out, lse) in enumerate(results):
        for b in range(WL.B):
            r = ref[li][(b, 0)]
            assert set(idx[b, 0][idx[b, 0] >= 0].tolist()) == set(r["idx"][r["idx"] >= 0].tolist()), (li, b)
            o = r["out"].astype(np.float64)
            rms = np.sqrt((o ** 2).mean(axis=-1))
            err = np.abs(out[b, 0].astype(np.float64) - o).max(axis=-1)
            assert np.all(err <= 2e-3 * rms), (li, b, float((err / rms).max()))
            assert np.allclose(lse[b, 0], r["lse"], rtol=1e-5, atol=1e-5), (li, b)


def test_slice_rows_partition():
    for L in (1, 7, 8, 3000, 4099, 1 << 20):
        for G in (1, 2, 3, 8):
            spans = [CS.slice_rows(L, G, g) for g in range(G)]
            assert spans[0][0] == 0 and spans[-1][1] == L
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0 and a0 <= a1
            assert all(lo % 8 == 0 for lo, _ in spans)


def test_two_gloo_ranks_match_the_whole_sequence():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        check_against_whole_sequence(out[rank])
    # both ranks hold the same merged result
    for a, b in zip(out[0], out[1]):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("world", [1, 3])
def test_in_process_ranks(world):
    """The same split with the ranks' phases run in turn in one process (the
    exchange is a concatenation), for one and three slices."""
    parts_results = []
    lat, ik, layers = _inputs()
    parts = []
    for g in range(world):
        lo, hi = CS.slice_rows(WL.L, world, g)
        cache = oracle.Cache(WL.B, hi - lo, WL.D, WL.DI)
        cache.append(lat[:, lo:hi].numpy(), ik[:, lo:hi].numpy())
        parts.append(CS.Part(cache, lo, hi - lo))
    prev = None
    for li, mode in enumerate(WL.layers):
        inp = layers[li]
        if mode != W.REUSE:
            pairs = [CS.local_pairs(p, inp["iq"], inp["w"], WL.K, OracleOps) for p in parts]
            prev = CS.global_selection([s for s, _ in pairs], [i for _, i in pairs], WL.K, OracleOps)
        partial = [CS.local_attention(p, inp["q"], prev, WL.scale, OracleOps) for p in parts]
        out, lse = CS.merge([o for o, _ in partial], [l for _, l in partial], OracleOps)
        parts_results.append((prev.numpy(), out.numpy(), lse.numpy()))
    check_against_whole_sequence(parts_results)
