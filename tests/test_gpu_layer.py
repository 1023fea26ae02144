"""a7 on the GPU: whole CSA2 layers and mode chains through csa_layer_step,
against the oracle chain on the same seeded inputs.

Small workloads are checked on every query; the full-size workloads (the
launch configuration the benchmark times) are checked on sampled sequences,
for which the oracle runs the whole chain on that sequence's rows.  Every
layer's selection is checked against the oracle's, and every query's attention
output against the oracle's attention over the rows the GPU selected (which
are the oracle's own rows unless the two differ by a near tie).
"""
import os

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import check_chain, device_cache, need_gpu

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))


def run_gpu_chain(wl, seed, cache):
    swa = B.Swa(W.local_rows(wl, seed, device="cuda"), wl.window) if wl.window else None
    w_ik = W.ikey_projection(wl, seed, device="cuda") if wl.project else None
    layers, prev, pool = [], None, None
    for li, mode in enumerate(wl.layers):
        inp = W.layer_inputs(wl, seed, li, device="cuda")
        app = W.append_rows(wl, seed, device="cuda") if (li == 0 and wl.n_append) else None
        la = B.LayerArgs(cache, mode, inp["q"], wl.K, wl.scale, iq=inp["iq"], w=inp["w"],
                         idx=prev if mode == W.REUSE else None,
                         rows_new=app["rows"] if app else None,
                         ikeys_new=app["ikeys"] if (app and not wl.project) else None,
                         w_ik=w_ik if app else None,
                         pool_in=pool if mode == W.REINDEX else None, pool_blocks=wl.pool_blocks,
                         make_pool=(mode == W.FULL and wl.pool_blocks > 0 and pool is None), swa=swa)
        B.csa_layer_step(cache, la)
        if mode != W.REUSE:
            prev = la.idx
        if la.pool_out is not None:
            pool = la.pool_out
        layers.append(la)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    return layers


SMALL = [
    W.WORKLOADS["tiny_full"],
    W.Workload("chain_small", B=2, L=5003, H=16, D=256, HI=16, DI=128, K=300,
               layers=(W.FULL, W.REINDEX, W.REINDEX, W.REUSE, W.REUSE)),
    W.Workload("hier_small", B=1, L=40000, H=64, D=512, HI=64, DI=128, K=512,
               layers=(W.FULL, W.REINDEX, W.REINDEX, W.REUSE), pool_blocks=128, planted=64),
    W.Workload("verify_small", B=3, L=3000, H=8, D=128, HI=32, DI=64, K=700, P=6, n_append=6),
    W.Workload("chain_swa_small", B=3, L=4000, H=32, D=512, HI=16, DI=128, K=512, P=2, outlier_channels=5,
               layers=(W.FULL, W.REINDEX, W.REUSE), window=128),
    W.Workload("verify_project_small", B=3, L=3000, H=8, D=256, HI=32, DI=64, K=700, P=6, n_append=6,
               project=True),
    W.Workload("chain_mx_small", B=2, L=5002, H=16, D=256, HI=16, DI=128, K=300, P=2, n_append=2,
               layers=(W.FULL, W.REINDEX, W.REUSE), key_format="mxfp4"),
    W.Workload("hier_mx_small", B=1, L=40000, H=64, D=512, HI=64, DI=128, K=512,
               layers=(W.FULL, W.REINDEX, W.REINDEX, W.REUSE), pool_blocks=128, key_format="mxfp4"),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_small_workloads_every_query(wl):
    need_gpu()
    cache, lat, ik = device_cache(wl, seed=0)
    gpu = run_gpu_chain(wl, 0, cache)
    check_chain(wl, 0, gpu, lat, ik, list(range(wl.B)), threads=THREADS)
    if wl.planted:
        off = W.planted_offset(wl, 0)
        for la in gpu:
            sel = set(la.idx[0, 0].cpu().tolist())
            assert set(range(off, off + wl.planted)) <= sel


FULL_SIZE = [("full_64k", [0, 5]), ("chain_128k", [17]), ("hier_1m", [0]), ("verify_append_32k", [40]),
             ("full_64k_swa", [3]), ("verify_project_32k", [11]), ("full_64k_mx", [2]), ("chain_128k_mx", [9])]


@pytest.mark.slow
@pytest.mark.parametrize("name,seqs", FULL_SIZE, ids=[n for n, _ in FULL_SIZE])
def test_full_size_sampled(name, seqs):
    need_gpu()
    wl = W.WORKLOADS[name]
    cache, lat, ik = device_cache(wl, seed=0)
    gpu = run_gpu_chain(wl, 0, cache)
    check_chain(wl, 0, gpu, lat, ik, seqs, threads=THREADS)
    # property at every query: selections are valid, sorted, unique, and in range
    for la in gpu:
        idx = la.idx.cpu().numpy()
        assert idx.max() < wl.length_after_append
        n = (idx >= 0).sum(axis=-1)
        assert np.all(n == min(wl.K, wl.L))
