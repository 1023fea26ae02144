"""MXFP4 indexer keys on the GPU: keys copied as given, scores over a full scan
and over a pool against the oracle's MXFP4 scores, and keys projected into
MXFP4 against the oracle's exactly rounded projection.

"G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache entries, and why
they're safe": 128 values x 4 bits + one 8-bit scale per 32 values = 68 B.
"""
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


def compare(gpu, ora, iq, w, keys, what):
    """fp32 against double: |err| <= 1e-5 x sum_h w_h sum_d |q_hd k_d|."""
    kc, ks = oracle.mx_unpack(keys, iq.shape[1])
    k = np.abs(oracle.mx_dequantize(kc, ks))
    bound = k @ np.abs(e4m3_f64(iq)).T @ np.abs(w.astype(np.float64))
    err = np.abs(gpu.astype(np.float64) - ora.astype(np.float64))
    assert np.all(err <= 1e-5 * bound + 1e-30), (what, float((err / np.maximum(bound, 1e-30)).max()))


def test_keys_are_copied_as_given():
    need_gpu()
    wl = W.Workload("t", B=2, L=300, H=4, D=128, HI=4, DI=128, K=8, key_format="mxfp4")
    cache, _, ik = device_cache(wl, seed=71)
    torch.cuda.synchronize()
    assert torch.equal(cache.packed_keys()[:, : wl.L].cpu(), ik.cpu())


@pytest.mark.parametrize("HI,P", [(4, 1), (64, 1), (16, 3)])
def test_full_scan_scores(HI, P):
    need_gpu()
    wl = W.Workload("t", B=2, L=3004, H=4, D=128, HI=HI, DI=128, K=8, P=P, key_format="mxfp4")
    cache, _, ik = device_cache(wl, seed=72)
    inp = W.layer_inputs(wl, 72, 0, device="cuda")
    scores = B.csa_index_score(cache, inp["iq"], inp["w"])
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    s = scores.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        for p in range(P):
            L = wl.L - P + 1 + p
            ora = oracle.index_scores_mx(iqh[b, p], wh[b, p], ikh[b], np.arange(L))
            compare(s[b, p, :L], ora, iqh[b, p], wh[b, p], ikh[b, :L], (b, p))


def test_scales_outside_the_written_range_apply_exactly():
    """Block scales the library never writes (bytes 100..150, X = -27..23) are
    applied as 2^(byte - 127) by the block-scaled MMA, as the oracle decodes them."""
    need_gpu()
    Bn, L, DI, HI = 2, 1100, 128, 16
    wl = W.Workload("t", B=Bn, L=L, H=4, D=128, HI=HI, DI=DI, K=8, key_format="mxfp4")
    cache = B.Cache(Bn, L, 128, DI, device="cuda", key_format="mxfp4")
    keys = W.random_mx_keys(Bn * L, DI, "cuda", 77).view(Bn, L, -1)
    keys[..., DI // 2:] = W.random_ints((Bn, L, DI // 32), 100, 151, seed=78).to(torch.uint8).cuda()
    B.csa_quantize_append(cache, W.random_bf16_bits((Bn, L, 128), seed=79, device="cuda"), keys)
    inp = W.layer_inputs(wl, 77, 0, device="cuda")
    scores = B.csa_index_score(cache, inp["iq"], inp["w"])
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    s = scores.cpu().numpy()
    ikh, iqh, wh = keys.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(Bn):
        ora = oracle.index_scores_mx(iqh[b, 0], wh[b, 0], ikh[b], np.arange(L))
        compare(s[b, 0, :L], ora, iqh[b, 0], wh[b, 0], ikh[b], b)


def test_pool_scores():
    need_gpu()
    wl = W.Workload("t", B=2, L=2004, H=4, D=128, HI=16, DI=128, K=8, key_format="mxfp4")
    cache, _, ik = device_cache(wl, seed=73)
    inp = W.layer_inputs(wl, 73, 0, device="cuda")
    nb = (wl.L + 7) // 8
    pool = np.full((wl.B, 1, 40), -1, np.int32)
    pool[0, 0, :37] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=3).numpy().argsort()[:37])
    pool[1, 0, :40] = np.sort(W.random_ints((nb,), 0, 1 << 30, seed=4).numpy().argsort()[:39].tolist() + [nb - 1])
    scores = B.csa_index_score(cache, inp["iq"], inp["w"], pool=torch.from_numpy(pool).cuda())
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    s = scores.cpu().numpy()
    ikh, iqh, wh = ik.cpu().numpy(), inp["iq"].cpu().numpy(), inp["w"].cpu().numpy()
    for b in range(wl.B):
        rows, valid = oracle.pool_rows(pool[b, 0], wl.L)
        v = valid.astype(bool)
        ora = oracle.index_scores_mx(iqh[b, 0], wh[b, 0], ikh[b], rows)
        compare(s[b, 0, :320][v], ora[v], iqh[b, 0], wh[b, 0], ikh[b, rows[v]], b)


def test_projected_mx_keys_match_oracle():
    """GPU sums are fp32: a block may take the other exponent where its exact
    largest magnitude lies within fp32 summation error of a power of two, and a
    code may differ where the exact value lies within it of an E2M1 midpoint."""
    need_gpu()
    D, DI, Bn, n_new = 512, 128, 3, 13
    cache = B.Cache(Bn, 40, D, DI, device="cuda", key_format="mxfp4")
    rows = W.random_bf16_bits((Bn, n_new, D), seed=74, device="cuda", std=2.0)
    wf = torch.randn((D, DI), generator=torch.Generator().manual_seed(75)) / D ** 0.5
    w_bits = wf.to(torch.bfloat16).view(torch.int16)
    B.csa_device_status()
    B.csa_quantize_append_project(cache, rows, w_bits.cuda())
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    got = cache.packed_keys()[:, :n_new].cpu().numpy()
    rb = rows.cpu().numpy()
    wb = w_bits.numpy().view(np.uint16)
    wd = wf.to(torch.bfloat16).to(torch.float64).numpy()
    odd = 0
    for b in range(Bn):
        codes, scales = oracle.quantize_rows(rb[b])
        ref = oracle.project_ikeys_mx(codes, scales, wb)
        v = oracle.dequantize_rows(codes, scales)
        exact, mag = v @ wd, np.abs(v) @ np.abs(wd)
        tol = 4 * D * 2.0 ** -24 * mag
        gc, gs = oracle.mx_unpack(got[b], DI)
        rc, rs = oracle.mx_unpack(ref, DI)
        for r in range(n_new):
            for blk in range(DI // 32):
                sl = slice(blk * 32, (blk + 1) * 32)
                if gs[r, blk] != rs[r, blk]:
                    amax = np.abs(exact[r, sl]).max()
                    edge = 2.0 ** (max(int(gs[r, blk]), int(rs[r, blk])) - 127 + 2)
                    assert abs(amax - edge) <= tol[r, sl].max(), (b, r, blk)
                    odd += 1
                    continue
                gn = np.stack([gc[r, blk * 16:(blk + 1) * 16] & 0xF, gc[r, blk * 16:(blk + 1) * 16] >> 4], 1).ravel()
                rn = np.stack([rc[r, blk * 16:(blk + 1) * 16] & 0xF, rc[r, blk * 16:(blk + 1) * 16] >> 4], 1).ravel()
                X = int(rs[r, blk]) - 127
                for i in np.nonzero(gn != rn)[0]:
                    ch = blk * 32 + i
                    q = abs(exact[r, ch]) / 2.0 ** X
                    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
                    assert np.abs(mids - q).min() <= tol[r, ch] / 2.0 ** X, (b, r, ch)
                    odd += 1
    assert odd <= 3
