"""csa_sparse_attend_noalloc: the attention entry point for callers that cannot
allocate device memory (their memory belongs to a host framework's allocator or
a fixed arena, or their serving loop cannot afford an allocation mid-step).

It must give the same answer as csa_sparse_attend with a caller workspace, on
two calls in a row (the fixed scratch array keeps the first call's partials),
and must refuse a problem whose partials do not fit the fixed array.  This file
is collected last so that a run stopping at its first failure has already run
every other test.
"""

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import check_attention, device_cache, need_gpu

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = B.CSA_NOALLOC_SCRATCH_BYTES


def test_noalloc_matches_workspace_call_twice():
    need_gpu()
    wl = W.Workload("noalloc", B=2, L=3000, H=16, D=256, HI=4, DI=64, K=1000, P=2)
    cache, _, _ = device_cache(wl, seed=31)
    q = W.layer_inputs(wl, 31, 0, device="cuda")["q"]
    idx = W.random_ints((wl.B, wl.P, wl.K), -1, wl.L - wl.P + 1, seed=32).to(torch.int32).cuda()
    ref_out, ref_lse = B.csa_sparse_attend(cache, q, idx, wl.scale)
    torch.cuda.synchronize()
    assert 0 < B.attend_workspace_size(cache, wl.P, wl.H, wl.K) <= SCRATCH_BYTES
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        B.csa_sparse_attend_noalloc(cache, q, idx, wl.scale, out, lse)
        torch.cuda.synchronize()
        assert B.csa_device_status() == 0
        check_attention(out.cpu().numpy(), ref_out.cpu().numpy(), ("call", call))
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-6, atol=1e-6)


def test_noalloc_ten_queries_with_partials_in_memory():
    """10 queries of 64 heads x 512 dims at K = 2048: 11 splits per query, more
    than a cluster holds, so the partials go through the scratch array (14.5 MB
    of its 17 MiB)."""
    need_gpu()
    wl = W.Workload("noalloc10", B=10, L=6000, H=64, D=512, HI=4, DI=64, K=2048)
    cache, _, _ = device_cache(wl, seed=41)
    assert 0 < B.attend_workspace_size(cache, wl.P, wl.H, wl.K) <= SCRATCH_BYTES
    q = W.layer_inputs(wl, 41, 0, device="cuda")["q"]
    idx = W.random_ints((wl.B, wl.P, wl.K), -1, wl.L, seed=42).to(torch.int32).cuda()
    ref_out, ref_lse = B.csa_sparse_attend(cache, q, idx, wl.scale)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    B.csa_sparse_attend_noalloc(cache, q, idx, wl.scale, out, lse)
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    check_attention(out.cpu().numpy(), ref_out.cpu().numpy(), "10 queries")
    assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("Bn", [9, 13])
def test_noalloc_refuses_problems_larger_than_its_array(Bn):
    """9 queries (16 splits each) and 13 (11 each) of 64 heads x 512 dims at
    K = 2048 need more partials than the array holds, though 10 to 12 fit."""
    need_gpu()
    P, H, K = 1, 64, 2048
    cache = B.Cache(Bn, 64, 512, 128)
    assert B.attend_workspace_size(cache, P, H, K) > SCRATCH_BYTES
    q = torch.zeros((Bn, P, H, 512), dtype=torch.int16, device="cuda")
    idx = torch.full((Bn, P, K), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((Bn, P, H, 512), dtype=torch.float32, device="cuda")
    with pytest.raises(B.CsaError) as e:
        B.csa_sparse_attend_noalloc(cache, q, idx, 1.0, out)
    assert e.value.status == 5                   # CSA_ERR_WORKSPACE
    assert torch.all(out == 0)                   # nothing was launched
