"""a1 on the GPU: FP4 quantise-and-append, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import need_gpu

pytestmark = pytest.mark.gpu


def all_finite_bf16_bits():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    return bits[exp != 0xFF]


def run_append(rows_bits: np.ndarray, D: int, ikeys=None, cap_extra=0):
    Bn, n, _ = rows_bits.shape
    cache = B.Cache(Bn, n + cap_extra, D, 64)
    rows = torch.from_numpy(rows_bits.view(np.int16)).cuda()
    ik = torch.from_numpy(ikeys).cuda() if ikeys is not None else None
    B.csa_quantize_append(cache, rows, ik)
    torch.cuda.synchronize()
    return cache


def test_exhaustive_bf16_patterns_bit_exact():
    need_gpu()
    vals = all_finite_bf16_bits()
    pad = (-len(vals)) % 512
    v = np.concatenate([vals, np.zeros(pad, np.uint16)])
    # sorted order (groups of similar magnitude) and a seeded shuffle (mixed groups)
    perm = W.random_ints((len(v),), 0, 1 << 30, seed=7).numpy().argsort()
    rows = np.stack([v.reshape(-1, 512), v[perm].reshape(-1, 512)])
    cache = run_append(rows, 512)
    codes, scales = oracle.quantize_rows(rows)
    assert np.array_equal(cache.codes.cpu().numpy(), codes)
    assert np.array_equal(cache.scales.cpu().numpy(), scales)
    assert cache.lengths.cpu().tolist() == [rows.shape[1]] * 2


@pytest.mark.parametrize("D", [128, 512])
def test_workload_rows_and_outliers_bit_exact(D):
    need_gpu()
    wl = W.Workload("t", B=3, L=777, H=4, D=D, HI=4, DI=64, K=8, outlier_channels=5)
    rows = np.stack([W.cache_rows(wl, 1, b)[0].numpy() for b in range(3)]).view(np.uint16)
    rows[0, 5, :16] = 0                        # all-zero group
    rows[1, 7, 16:32] = 0x8000                 # all -0
    rows[2, 9, 0] = 0x4600                     # 8192: saturating group
    rows[2, 9, 1] = 0xC600
    cache = run_append(rows, D)
    codes, scales = oracle.quantize_rows(rows)
    assert np.array_equal(cache.codes.cpu().numpy(), codes)
    assert np.array_equal(cache.scales.cpu().numpy(), scales)


def test_append_positions_lengths_and_capacity():
    need_gpu()
    D, DI = 128, 64
    cache = B.Cache(2, 10, D, DI)
    r1 = W.random_bf16_bits((2, 4, D), 2, 1).cuda()
    k1 = W.random_e4m3_bytes((2, 4, DI), 2, 2).cuda()
    r2 = W.random_bf16_bits((2, 5, D), 2, 3).cuda()
    k2 = W.random_e4m3_bytes((2, 5, DI), 2, 4).cuda()
    B.csa_quantize_append(cache, r1, k1)
    B.csa_quantize_append(cache, r2, k2)
    assert B.csa_device_status() == 0
    assert cache.lengths.cpu().tolist() == [9, 9]
    allr = torch.cat([r1, r2], 1).cpu().numpy().view(np.uint16)
    codes, scales = oracle.quantize_rows(allr)
    assert np.array_equal(cache.codes[:, :9].cpu().numpy(), codes)
    assert np.array_equal(cache.scales[:, :9].cpu().numpy(), scales)
    assert np.array_equal(cache.ikeys[:, :9].cpu().numpy(), torch.cat([k1, k2], 1).cpu().numpy())
    assert not cache.codes[:, 9:].any()
    # a third append of 2 rows would pass capacity 10: sequences stay unchanged
    before = cache.codes.clone()
    B.csa_quantize_append(cache, r1[:, :2].contiguous(), None)
    assert B.csa_device_status() & B.CSA_DEV_CAPACITY
    assert cache.lengths.cpu().tolist() == [9, 9]
    assert torch.equal(before, cache.codes)
    assert B.csa_device_status() == 0          # cleared by the previous read
