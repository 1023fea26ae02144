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


# ---------------------------------------------------------------------------
# Whole chains
# ---------------------------------------------------------------------------

def oracle_inputs(wl: W.Workload, seed: int, lat, ik, seqs, threads: int):
    """Oracle cache of the listed sequences (host copies of the same draws, the
    step's appended rows included) and each layer's inputs for them."""
    cache = oracle.Cache(len(seqs), wl.capacity, wl.D, wl.DI, key_format=wl.key_format)
    w_ik = W.ikey_projection(wl, seed, device="cuda").cpu().numpy() if wl.project else None
    project = oracle.project_ikeys_mx if wl.key_format == "mxfp4" else oracle.project_ikeys

    def keys(rows_bits, given):
        # projected workloads: the oracle projects the keys itself, from its own quantisation
        if not wl.project:
            return given
        return np.stack([project(*oracle.quantize_rows(r), w_ik) for r in rows_bits])

    lat_s = lat[seqs].cpu().numpy()
    cache.append(lat_s, keys(lat_s, None if ik is None else ik[seqs].cpu().numpy()), threads=threads)
    if wl.n_append:
        app = W.append_rows(wl, seed, device="cuda")
        rows_s = app["rows"][seqs].cpu().numpy()
        cache.append(rows_s, keys(rows_s, app["ikeys"][seqs].cpu().numpy()))
    inputs = []
    for li in range(len(wl.layers)):
        inp = W.layer_inputs(wl, seed, li, device="cuda")
        inputs.append({k: v[seqs].cpu().numpy() for k, v in inp.items()})
    swa = (W.local_rows(wl, seed, device="cuda")[seqs].cpu().numpy(), wl.window) if wl.window else None
    return cache, inputs, swa


def oracle_attend_unit(cache, j: int, p: int, q_bits, idx, wl: W.Workload, swa=None):
    """The oracle's attention (joint with the local window when swa is given)
    of oracle sequence j, position p over the selection idx."""
    if swa is None:
        return oracle.attend(q_bits, cache.codes[j], cache.scales[j], idx, wl.scale)
    rows_b, window = swa[0][j], swa[1]
    lo, hi = oracle.swa_window(rows_b.shape[0], wl.P, p, window)
    return oracle.attend_swa(q_bits, cache.codes[j], cache.scales[j], idx, rows_b, lo, hi, wl.scale)


def check_chain(wl: W.Workload, seed: int, gpu_layers, lat, ik, seqs, threads: int = 1) -> int:
    """Checks every layer of a chain the GPU ran, on the listed sequences, at
    every query position.

    Several selections can be correct where scores tie to within the top-K
    tolerance, so the GPU's choices are first checked against the oracle's
    (check_topk), and the oracle then continues from the GPU's validated
    choices: Reindex layers rescore the GPU's pool, Reuse layers attend over
    the GPU's previous selection, and every attention output is compared with
    the oracle's attention over the very rows the GPU selected.  Returns the
    number of (layer, query) units whose selection differed by a near tie."""
    cache, inputs, swa = oracle_inputs(wl, seed, lat, ik, seqs, threads)
    units = [(j, p) for j in range(len(seqs)) for p in range(wl.P)]
    prev, pool, near_ties = None, None, 0
    for li, mode in enumerate(wl.layers):
        g = gpu_layers[li]
        gi = g.idx.cpu().numpy()
        go = g.out.cpu().numpy()
        r = oracle.run_layer(cache, mode, inputs[li], wl.K, wl.scale, wl.P,
                             prev_idx=prev if mode == W.REUSE else None,
                             pool_in=pool if mode == W.REINDEX else None,
                             pool_keep=wl.pool_blocks if (mode == W.FULL and pool is None) else 0,
                             units=units, threads=min(threads, len(units)), score_threads=threads, swa=swa)
        for (j, p) in units:
            b = seqs[j]
            ru = r[(j, p)]
            what = (wl.name, li, b, p)
            ascending_then_padding(gi[b, p])
            equal = True
            if mode != W.REUSE:
                if "rows" in ru:
                    ok = ru["valid"] > 0
                    by_row = dict(zip(ru["rows"][ok].tolist(), ru["scores"][ok].tolist()))
                    scores_of = lambda rows, m=by_row: np.array([m[int(x)] for x in rows], np.float32)
                else:
                    scores_of = lambda rows, s=ru["scores"]: s[rows]
                equal = check_topk(gi[b, p], ru["idx"], scores_of, wl.K, what)
            if "pool" in ru:
                bm = oracle.block_max(ru["scores"])
                check_topk(g.pool_out.cpu().numpy()[b, p], ru["pool"], lambda blocks, s=bm: s[blocks],
                           wl.pool_blocks, what + ("pool",))
            if equal:
                ref = ru["out"]
            else:
                near_ties += 1
                ref, _ = oracle_attend_unit(cache, j, p, inputs[li]["q"][j, p], gi[b, p], wl, swa)
            check_attention(go[b, p], ref, what)
        if mode != W.REUSE:
            prev = {(j, p): gi[seqs[j], p].astype(np.int64) for (j, p) in units}
        if mode == W.FULL and wl.pool_blocks and pool is None:
            gp = gpu_layers[li].pool_out.cpu().numpy()
            pool = {(j, p): gp[seqs[j], p].astype(np.int64) for (j, p) in units}
    return near_ties
