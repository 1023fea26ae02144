"""The local window joined to the sparse attention on the GPU (csa_sparse_attend_swa
and csa_layer_step with a window) against the oracle's joint softmax.

The window rows are FP8 E4M3 bytes drawn once and given to both sides; the
oracle quantises the same bf16 cache rows itself and decodes the window bytes
itself.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import check_attention, check_topk, device_cache, need_gpu

pytestmark = pytest.mark.gpu


def selection(wl, seed):
    idx = W.random_ints((wl.B, wl.P, wl.K), 0, wl.L, seed=seed).to(torch.int32)
    if wl.K > 1:
        idx[..., ::5] = -1                             # padding entries are skipped
    return idx


def check_units(out, lse, q, lat, idx, local, lens, wl, units):
    qh, ih, wh = q.cpu().numpy(), idx.numpy(), local.cpu().numpy()
    done = {}
    for b, p in units:
        if b not in done:
            done[b] = oracle.quantize_rows(lat[b].cpu().numpy())
        codes, scales = done[b]
        lo, hi = oracle.swa_window(lens[b], wl.P, p, wl.window)
        o, l = oracle.attend_swa(qh[b, p], codes, scales, ih[b, p], wh[b], lo, hi, wl.scale)
        check_attention(out[b, p].cpu().numpy(), o, (b, p))
        assert np.allclose(lse[b, p].cpu().numpy(), l, rtol=1e-5, atol=1e-5), (b, p)


# Split plans covered (one window split added to the selection's splits): a
# cluster of 5 (1 query), 16 + 1 splits merged through global memory (2
# queries), a cluster of 3 with a different window per position (6 queries), a
# cluster of 7 (20 queries), a window of 16 tiles with ragged local lengths
# (windows of 1 and 2 rows at the start of a sequence), one selected row
# beside a full window, and 11 + 1 splits through the merge kernel.
@pytest.mark.parametrize("H,D,K,Bn,P,window,lens", [
    (16, 128, 256, 1, 1, 128, None),
    (64, 512, 2048, 2, 1, 128, None),
    (7, 256, 100, 2, 3, 50, None),
    (64, 512, 2048, 20, 1, 128, None),
    (32, 256, 64, 3, 2, 1000, (2, 700, 1001)),
    (64, 512, 1, 1, 1, 128, None),
    (64, 512, 2048, 9, 1, 128, None),
])
def test_joint_softmax_matches_oracle(H, D, K, Bn, P, window, lens):
    need_gpu()
    wl = W.Workload("t", B=Bn, L=5000, H=H, D=D, HI=4, DI=64, K=K, P=P, outlier_channels=5, window=window)
    cache, lat, _ = device_cache(wl, seed=31)
    q = W.layer_inputs(wl, 31, 0, device="cuda")["q"]
    idx = selection(wl, 32)
    n = max(lens) if lens else window + P - 1
    local = W.local_rows(wl, 33, device="cuda", n=n)
    lengths = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens else None
    B.csa_device_status()
    out, lse = B.csa_sparse_attend_swa(cache, q, idx.cuda(), wl.scale, B.Swa(local, window, lengths))
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    L = list(lens) if lens else [n] * Bn
    check_units(out, lse, q, lat, idx, local, L, wl, [(b, p) for b in range(Bn) for p in range(P)])


def test_one_wave_of_queries_sampled():
    """148 queries: the selection takes one split and the window one more (a
    cluster of 2 per query); a sample of the queries is checked."""
    need_gpu()
    wl = W.Workload("t", B=148, L=3000, H=64, D=512, HI=4, DI=64, K=2048, outlier_channels=5, window=128)
    cache, lat, _ = device_cache(wl, seed=34)
    q = W.layer_inputs(wl, 34, 0, device="cuda")["q"]
    idx = selection(wl, 35)
    local = W.local_rows(wl, 36, device="cuda")
    out, lse = B.csa_sparse_attend_swa(cache, q, idx.cuda(), wl.scale, B.Swa(local, wl.window))
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    check_units(out, lse, q, lat, idx, local, [local.shape[1]] * wl.B, wl, [(0, 0), (73, 0), (147, 0)])


def test_window_alone_and_bad_lengths():
    """An empty selection leaves the window alone; a local length outside
    [P, n] raises the bad-index bit and leaves that sequence's window empty."""
    need_gpu()
    wl = W.Workload("t", B=3, L=300, H=8, D=128, HI=4, DI=64, K=16, P=2, window=20)
    cache, lat, _ = device_cache(wl, seed=37)
    q = W.layer_inputs(wl, 37, 0, device="cuda")["q"]
    idx = torch.full((3, 2, 16), -1, dtype=torch.int32)
    idx[1, :, :3] = torch.tensor([4, 9, 200], dtype=torch.int32)
    local = W.local_rows(wl, 38, device="cuda", n=40)
    lengths = torch.tensor([30, 1, 41], dtype=torch.int32, device="cuda")   # 1 < P, 41 > n
    B.csa_device_status()
    out, lse = B.csa_sparse_attend_swa(cache, q, idx.cuda(), wl.scale, B.Swa(local, wl.window, lengths))
    assert B.csa_device_status() & B.CSA_DEV_BAD_INDEX
    check_units(out, lse, q, lat, idx, local, [30, 0, 0], wl, [(0, 0), (0, 1)])
    codes, scales = oracle.quantize_rows(lat[1].cpu().numpy())
    for p in range(2):
        o, l = oracle.attend(q[1, p].cpu().numpy(), codes, scales, idx[1, p].numpy(), wl.scale)
        check_attention(out[1, p].cpu().numpy(), o, (1, p))
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))


def test_no_window_is_plain_sparse_attention():
    need_gpu()
    wl = W.Workload("t", B=2, L=2000, H=16, D=256, HI=4, DI=64, K=300)
    cache, _, _ = device_cache(wl, seed=39)
    q = W.layer_inputs(wl, 39, 0, device="cuda")["q"]
    idx = selection(wl, 40).cuda()
    o1, l1 = B.csa_sparse_attend(cache, q, idx, wl.scale)
    o2, l2 = B.csa_sparse_attend_swa(cache, q, idx, wl.scale, None)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("mode", [W.FULL, W.REUSE])
def test_layer_step_with_window(mode):
    """csa_layer_step with a window: Full selects (checked against the oracle's
    top-K) and attends jointly; Reuse attends jointly over a given selection."""
    need_gpu()
    wl = W.Workload("t", B=2, L=3000, H=16, D=256, HI=8, DI=64, K=256, P=2, outlier_channels=5, window=128)
    cache, lat, ik = device_cache(wl, seed=41)
    inp = W.layer_inputs(wl, 41, 0, device="cuda")
    local = W.local_rows(wl, 42, device="cuda")
    swa = B.Swa(local, wl.window)
    given = selection(wl, 43)
    la = B.LayerArgs(cache, mode, inp["q"], wl.K, wl.scale, iq=inp["iq"], w=inp["w"],
                     idx=given.cuda() if mode == W.REUSE else None, swa=swa)
    B.csa_layer_step(cache, la)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    qh, wh = inp["q"].cpu().numpy(), local.cpu().numpy()
    for b in range(wl.B):
        codes, scales = oracle.quantize_rows(lat[b].cpu().numpy())
        for p in range(wl.P):
            if mode == W.FULL:
                rows = np.arange(oracle.visible_length(wl.L, wl.P, p), dtype=np.int64)
                s = oracle.index_scores(inp["iq"][b, p].cpu().numpy(), inp["w"][b, p].cpu().numpy(),
                                        ik[b].cpu().numpy(), rows)
                sel = oracle.topk(s, wl.K)
                if not check_topk(la.idx[b, p].cpu().numpy(), sel, lambda r, s=s: s[r], wl.K, (b, p)):
                    # a near-tie swap, which is a correct selection too: the
                    # reference is the attention over the rows the GPU chose
                    sel = la.idx[b, p].cpu().numpy().astype(np.int64)
            else:
                sel = given[b, p].numpy()
            lo, hi = oracle.swa_window(local.shape[1], wl.P, p, wl.window)
            o, l = oracle.attend_swa(qh[b, p], codes, scales, sel, wh[b], lo, hi, wl.scale)
            check_attention(la.out[b, p].cpu().numpy(), o, (b, p))
            assert np.allclose(la.lse[b, p].cpu().numpy(), l, rtol=1e-5, atol=1e-5), (b, p)
