"""Shared helpers of the GPU parity tests: device caches built through the C ABI,
host copies for the oracle, and the acceptance rules.

Acceptance (same on every test):
* FP4 codes and scale bytes: bit-exact.
* top-K index sets: exact, except members of the symmetric difference whose
  oracle score is within 1e-5 relative of the oracle's K-th score (near ties).
* attention: max |gpu - oracle| <= 2e-3 x RMS of that oracle output row.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_compressed_sparse_append_b300 import binding as B
from fp4_compressed_sparse_append_b300 import build as BUILD
from fp4_compressed_sparse_append_b300 import workloads as W

TOPK_REL = 1e-5
ATT_REL = 2e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BUILD.build()
    B.lib()


def device_cache(wl: W.Workload, seed: int, device="cuda"):
    """Draw the workload's cached rows on the device, quantise-append them through
    the C ABI.  Returns (cache, latents [B, L, D] int16 bits, ikeys [B, L, DI] u8), on the device."""
    cache = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device=device, key_format=wl.key_format)
    lat = torch.empty((wl.B, wl.L, wl.D), dtype=torch.int16, device=device)
    ik = torch.empty((wl.B, wl.L, W.key_bytes(wl)), dtype=torch.uint8, device=device)
    for b in range(wl.B):
        lat[b], ik[b] = W.cache_rows(wl, seed, b, device=device)
    if wl.project:
        # keys projected from the stored rows (the drawn keys are not used)
        B.csa_quantize_append_project(cache, lat, W.ikey_projection(wl, seed, device=device))
        ik = None          # the oracle projects its own keys
    else:
        B.csa_quantize_append(cache, lat, ik)
    return cache, lat, ik


def check_topk(gpu_idx, ora_idx, ora_scores_of, K, what=""):
    """gpu_idx/ora_idx: int arrays (with -1 padding).  ora_scores_of: callable
    mapping row ids -> oracle fp32 scores.  Returns True if the sets are equal."""
    g = set(int(x) for x in gpu_idx if x >= 0)
    o = set(int(x) for x in ora_idx if x >= 0)
    assert len(g) == len(o), (what, len(g), len(o))
    if g == o:
        return True
    diff = np.array(sorted(g ^ o), np.int64)
    kth = float(np.min(ora_scores_of(np.array(sorted(o), np.int64))))
    ds = ora_scores_of(diff).astype(np.float64)
    bad = np.abs(ds - kth) > TOPK_REL * max(abs(kth), 1e-30)
    assert not bad.any(), (what, diff[bad][:8], ds[bad][:8], kth)
    return False


def check_attention(gpu_out, ora_out, what=""):
    """Row-wise: max abs error <= 2e-3 x RMS of the oracle row.  Arrays [..., D]."""
    g = np.asarray(gpu_out, np.float64)
    o = np.asarray(ora_out, np.float64)
    rms = np.sqrt((o ** 2).mean(axis=-1))
    err = np.abs(g - o).max(axis=-1)
    ok = err <= ATT_REL * rms
    empty = rms == 0
    ok |= empty & (err == 0)
    assert ok.all(), (what, float((err / np.maximum(rms, 1e-30)).max()))
    return float((err / np.maximum(rms, 1e-30))[~empty].max()) if (~empty).any() else 0.0


def ascending_then_padding(idx_row):
    v = np.asarray(idx_row)
    n = int((v >= 0).sum())
    assert np.all(v[n:] == -1)
    assert np.all(np.diff(v[:n]) > 0)
