"""Indexer keys projected from the stored rows (csa_quantize_append_project) on
the GPU against the oracle.

The oracle quantises the same bf16 rows itself and projects its own stored
entries exactly (double, rounded once).  The GPU sums in fp32, so a key may
differ by one code where the exact product lies within fp32 summation error of
the midpoint between two E4M3 values; every other byte must be equal.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import workloads as W
from gpu_common import need_gpu

pytestmark = pytest.mark.gpu


def e4m3_values(b):
    return torch.from_numpy(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def check_keys(gpu_ik, rows_bits, w_bits, what=""):
    """gpu_ik [n, DI] vs the oracle's projection of rows_bits [n, D] by w_bits [D, DI]."""
    codes, scales = oracle.quantize_rows(rows_bits)
    ref = oracle.project_ikeys(codes, scales, w_bits)
    diff = np.nonzero(gpu_ik != ref)
    if len(diff[0]) == 0:
        return 0
    v = oracle.dequantize_rows(codes, scales)                                    # exact
    wf = torch.from_numpy(np.ascontiguousarray(w_bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    exact = v @ wf                                                               # exact for these sizes
    mag = np.abs(v) @ np.abs(wf)
    D = v.shape[1]
    for r, j in zip(*diff):
        a, b = sorted(e4m3_values(np.array([gpu_ik[r, j] & 0x7F, ref[r, j] & 0x7F], np.uint8)))
        mid = (a + b) / 2
        tol = 4 * D * 2.0 ** -24 * mag[r, j]
        assert (gpu_ik[r, j] ^ ref[r, j]) & 0x80 == 0, (what, r, j)             # same sign
        assert abs(abs(exact[r, j]) - mid) <= tol, (what, r, j, exact[r, j], gpu_ik[r, j], ref[r, j])
    return len(diff[0])


@pytest.mark.parametrize("D,DI,n_new,w_scale", [(128, 32, 1, 1.0), (256, 64, 6, 1.0), (512, 128, 13, 1.0),
                                               (512, 128, 8, 300.0)])
def test_projected_keys_match_oracle(D, DI, n_new, w_scale):
    need_gpu()
    Bn, L0 = 3, 40
    cache = B.Cache(Bn, L0 + n_new + 5, D, DI, device="cuda")
    old = W.random_bf16_bits((Bn, L0, D), seed=51, device="cuda")
    old_ik = W.random_e4m3_bytes((Bn, L0, DI), seed=52, device="cuda")
    B.csa_quantize_append(cache, old, old_ik)
    new = W.random_bf16_bits((Bn, n_new, D), seed=53, device="cuda", std=2.0)
    wf = torch.randn((D, DI), generator=torch.Generator().manual_seed(54)) / D ** 0.5 * w_scale
    w_bits = wf.to(torch.bfloat16).view(torch.int16)
    B.csa_device_status()
    B.csa_quantize_append_project(cache, new, w_bits.cuda())
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    assert torch.all(cache.lengths.cpu() == L0 + n_new)
    assert torch.equal(cache.ikeys[:, :L0].cpu(), old_ik.cpu())                  # earlier keys untouched
    nb = new.cpu().numpy()
    codes, scales = oracle.quantize_rows(nb)
    assert np.array_equal(cache.codes[:, L0:L0 + n_new].cpu().numpy(), codes)
    assert np.array_equal(cache.scales[:, L0:L0 + n_new].cpu().numpy(), scales)
    gik = cache.ikeys[:, L0:L0 + n_new].cpu().numpy()
    flips = 0
    for b in range(Bn):
        flips += check_keys(gik[b], nb[b], w_bits.numpy().view(np.uint16), (D, DI, b))
    assert flips <= max(1, gik.size // 2000)
    if w_scale > 100:
        assert np.any((gik & 0x7F) == 0x7E)                                      # saturated keys occur


def test_projection_respects_capacity():
    need_gpu()
    D, DI = 128, 64
    cache = B.Cache(2, 12, D, DI, device="cuda")
    B.csa_quantize_append(cache, W.random_bf16_bits((2, 8, D), seed=55, device="cuda"),
                          W.random_e4m3_bytes((2, 8, DI), seed=56, device="cuda"))
    before = cache.ikeys.clone()
    cache.lengths[1] = 10                                                        # 10 + 3 > capacity 12
    B.csa_device_status()
    w_bits = (torch.randn((D, DI), generator=torch.Generator().manual_seed(57)) / D ** 0.5).to(torch.bfloat16)
    B.csa_quantize_append_project(cache, W.random_bf16_bits((2, 3, D), seed=58, device="cuda"),
                                  w_bits.view(torch.int16).cuda())
    assert B.csa_device_status() & B.CSA_DEV_CAPACITY
    assert torch.equal(cache.ikeys[1], before[1]) and int(cache.lengths[1]) == 10
    assert int(cache.lengths[0]) == 11


def test_layer_step_projects_new_keys():
    """A Full step with w_ik appends the rows, projects their keys, and scores
    them: the new rows' keys equal a separate projected append's keys."""
    need_gpu()
    wl = W.Workload("t", B=2, L=500, H=8, D=256, HI=16, DI=64, K=64, P=2, n_append=2, project=True)
    caches = []
    for _ in range(2):
        c = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device="cuda")
        lat = torch.stack([W.cache_rows(wl, 61, b, device="cuda")[0] for b in range(wl.B)])
        B.csa_quantize_append_project(c, lat, W.ikey_projection(wl, 61, device="cuda"))
        caches.append(c)
    app = W.append_rows(wl, 61, device="cuda")
    inp = W.layer_inputs(wl, 61, 0, device="cuda")
    la = B.LayerArgs(caches[0], W.FULL, inp["q"], wl.K, wl.scale, iq=inp["iq"], w=inp["w"], rows_new=app["rows"],
                     w_ik=W.ikey_projection(wl, 61, device="cuda"))
    B.csa_layer_step(caches[0], la)
    B.csa_quantize_append_project(caches[1], app["rows"], W.ikey_projection(wl, 61, device="cuda"))
    torch.cuda.synchronize()
    assert B.csa_device_status() == 0
    for t in ("codes", "scales", "ikeys", "lengths"):
        assert torch.equal(getattr(caches[0], t), getattr(caches[1], t)), t
