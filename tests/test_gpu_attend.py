"""a5/a6 on the GPU: sparse attention over given selections against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import check_attention, device_cache, need_gpu

pytestmark = pytest.mark.gpu


def host_cache(cache):
    return cache.codes.cpu().numpy(), cache.scales.cpu().numpy()


# Split plans covered: a cluster of 2 and of 4 splits merged on chip (one
# query), 32 splits merged by the merge kernel (2 queries), one split (6 queries
# of 7 heads, 3 positions), clusters of 7 (20 queries) and of odd sizes whose
# last dim slice is shorter (29 and 21 queries at D = 384 and 256), 11 splits
# merged by the merge kernel with 48 heads at D = 384 (12 queries), 16 splits
# (8 queries, the 64K decode shape), and one split per query (160 queries, more
# queries than SMs).  Two cases use a logit scale of 1, where a later tile's
# maximum exceeds the running one by more than 2^8 and the accumulated output
# is rescaled.  Few queries split their heads into groups: 2 groups of 32
# heads (2 queries), 4 of 16 (one query, with 32 splits and with a cluster of
# 8), 2 of 16 (32 heads), and groups that are not a multiple of 16: 2 of 24
# (48 heads) and 2 of 20 (40 heads, 2 queries), whose query boxes reach into
# the next group's rows and past the last query.
CASES = [(16, 128, 256, 1, 1, None), (64, 512, 2048, 2, 1, None), (7, 256, 100, 2, 3, None),
         (64, 512, 1, 1, 1, None), (64, 512, 2048, 20, 1, None), (48, 384, 700, 12, 1, None),
         (64, 512, 2048, 8, 1, None), (8, 384, 320, 29, 1, None), (8, 256, 448, 21, 1, None),
         (32, 512, 4096, 1, 1, 1.0), (64, 128, 4096, 1, 1, 1.0), (64, 512, 512, 1, 1, None),
         (16, 128, 200, 160, 1, None), (48, 512, 2048, 1, 1, None), (40, 256, 1500, 2, 1, None)]


@pytest.mark.parametrize("H,D,K,Bn,P,scale", CASES)
def test_attention_matches_oracle(H, D, K, Bn, P, scale):
    need_gpu()
    wl = W.Workload("t", B=Bn, L=5000, H=H, D=D, HI=4, DI=64, K=K, P=P, outlier_channels=5)
    sc = wl.scale if scale is None else scale
    cache, lat, _ = device_cache(wl, seed=21)
    q = W.layer_inputs(wl, 21, 0, device="cuda")["q"]
    idx = W.random_ints((Bn, P, K), 0, wl.L, seed=22).to(torch.int32)
    idx[..., ::5] = -1                                 # padding entries are skipped
    if K > 2:
        idx[..., 1] = idx[..., 2]                      # a duplicated row counts twice
    out, lse = B.csa_sparse_attend(cache, q, idx.cuda(), sc)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    # the oracle quantises the same bf16 rows itself
    codes, scales = oracle.quantize_rows(lat.cpu().numpy())
    qh, ih = q.cpu().numpy(), idx.numpy()
    for b in range(Bn):
        for p in range(P):
            o, l = oracle.attend(qh[b, p], codes[b], scales[b], ih[b, p], sc)
            check_attention(out[b, p].cpu().numpy(), o, (b, p))
            assert np.allclose(lse[b, p].cpu().numpy(), l, rtol=1e-5, atol=1e-5)


def test_empty_selection_and_bad_index():
    need_gpu()
    wl = W.Workload("t", B=2, L=300, H=8, D=128, HI=4, DI=64, K=16)
    cache, lat, _ = device_cache(wl, seed=23)
    q = W.layer_inputs(wl, 23, 0, device="cuda")["q"]
    idx = torch.full((2, 1, 16), -1, dtype=torch.int32)
    idx[1, 0, :5] = torch.tensor([3, 299, 300, 5000, 7])     # 300 and 5000 are past the length
    B.csa_device_status()
    out, lse = B.csa_sparse_attend(cache, q, idx.cuda(), wl.scale)
    assert B.csa_device_status() & B.CSA_DEV_BAD_INDEX
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    codes, scales = oracle.quantize_rows(lat.cpu().numpy())
    o, _ = oracle.attend(q[1, 0].cpu().numpy(), codes[1], scales[1], np.array([3, 299, 7]), wl.scale)
    check_attention(out[1, 0].cpu().numpy(), o)
