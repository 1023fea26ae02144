"""CPU oracle for the CSA2 decode step over an FP4 global KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path never calls it and shares no code with it.

The arithmetic lives in ``csa_oracle.c`` (plain C, double precision, loaded
with ctypes); this file only marshals numpy arrays and composes the per-layer
modes in the order the pages give them:

* "G2C Brief - DeepSeek V4.1-Flash: a model designed around its KV cache",
  section "CSA2: most layers don't keep their own cache" (mode table): Full
  computes its own KV, indexer keys and selection; Reindex borrows the KV and
  indexer keys and re-scores with its own indexer query; Reuse borrows the KV
  and the last selection.  Every layer has its own query.
* same page, "The hierarchical indexer": the first Full layer also groups
  positions into blocks of 8, scores each block by its best member and keeps
  the top 2,048 blocks; later Reindex layers search only that pool.
* "DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section "The
  Paper": Reuse takes the KV from the last Full layer and the indices from the
  last Full or Reindex layer.

Parity pins for every function are in ``tests/test_oracle_*.py``.  The whole
composed step has no printed worked example on any page: its numbers are
"parity unpinned" beyond the per-function pins and the mode invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "libcsa_oracle.so")

FULL, REINDEX, REUSE = 0, 1, 2
POOL_BLOCK = 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_value.restype = dbl
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = dbl
        L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_value.restype = dbl
        L.oracle_e4m3_round_ratio.argtypes = [dbl, dbl]
        L.oracle_e4m3_round_ratio.restype = ctypes.c_uint8
        L.oracle_e2m1_round_ratio.argtypes = [dbl, dbl]
        L.oracle_e2m1_round_ratio.restype = ctypes.c_uint8
        L.oracle_quantize_rows.argtypes = [P, i64, i32, P, P]
        L.oracle_dequantize_rows.argtypes = [P, P, i64, i32, P]
        L.oracle_index_score.argtypes = [P, P, i32, i32, P, P, i64, P]
        L.oracle_topk.argtypes = [P, P, i64, i64, P]
        L.oracle_block_max.argtypes = [P, i64, i32, P]
        L.oracle_attend.argtypes = [P, i32, i32, dbl, P, P, P, i64, P, P]
        L.oracle_attend_swa.argtypes = [P, i32, i32, dbl, P, P, P, i64, P, i64, i64, P, P]
        L.oracle_project_ikeys.argtypes = [P, P, i64, i32, P, i32, P]
        L.oracle_mx_exponent.argtypes = [dbl]
        L.oracle_mx_exponent.restype = ctypes.c_int
        L.oracle_mx_quantize.argtypes = [P, i64, i32, P, P]
        L.oracle_mx_quantize.restype = None
        L.oracle_mx_dequantize.argtypes = [P, P, i64, i32, P]
        L.oracle_mx_dequantize.restype = None
        L.oracle_index_score_mx.argtypes = [P, P, i32, i32, P, P, P, i64, P]
        L.oracle_index_score_mx.restype = None
        L.oracle_project_ikeys_mx.argtypes = [P, P, i64, i32, P, i32, P, P]
        L.oracle_project_ikeys_mx.restype = None
        L.oracle_project_ikeys.restype = None
        L.oracle_e4m3_round.argtypes = [dbl]
        L.oracle_e4m3_round.restype = ctypes.c_uint8
        L.oracle_record_bytes.argtypes = [i32, i32, i32]
        L.oracle_record_bytes.restype = i64
        L.oracle_bytes_per_token.argtypes = [P, P, i32]
        L.oracle_bytes_per_token.restype = dbl
        L.oracle_cache_spill.argtypes = [P, P, P, i32, i64, i32, i32, i32, P, i64, i64, P]
        L.oracle_cache_spill.restype = None
        L.oracle_cache_reload.argtypes = [P, P, P, i32, i64, i32, i32, i32, P, P, i64]
        L.oracle_cache_reload.restype = ctypes.c_int
        for f in (L.oracle_quantize_rows, L.oracle_dequantize_rows, L.oracle_index_score,
                  L.oracle_topk, L.oracle_block_max, L.oracle_attend):
            f.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(x, dtype) -> np.ndarray:
    """Accept numpy arrays or CPU torch tensors; return a C-contiguous numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = np.asarray(x)
    dt = np.dtype(dtype)
    if a.dtype != dt:
        if a.dtype.kind in "iu" and dt.kind in "iu" and a.dtype.itemsize == dt.itemsize:
            a = a.view(dt)          # raw bits (e.g. bf16 bits held as int16)
        else:
            a = a.astype(dt)
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------
# Scalar formats
# --------------------------------------------------------------------------

def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(byte)


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits & 0xFFFF)


# --------------------------------------------------------------------------
# a1: quantise (+ append)
# --------------------------------------------------------------------------

def _chunks(n: int, threads: int):
    step = max(1, -(-n // max(1, threads)))
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def quantize_rows(x_bits, threads: int = 1) -> tuple:
    """bf16 bits [..., D] -> (codes uint8 [..., D/2], scales uint8 [..., D/16]).
    threads > 1 splits the rows over threads (the rows are independent)."""
    x = _np(x_bits, np.uint16)
    D = x.shape[-1]
    n = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    codes = np.zeros(x.shape[:-1] + (D // 2,), np.uint8)
    scales = np.zeros(x.shape[:-1] + (D // 16,), np.uint8)
    xf, cf, sf = x.reshape(n, D), codes.reshape(n, D // 2), scales.reshape(n, D // 16)

    def part(r):
        a, b = r
        lib().oracle_quantize_rows(_ptr(xf[a:b]), b - a, D, _ptr(cf[a:b]), _ptr(sf[a:b]))

    if threads > 1 and n > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, _chunks(n, threads)))
    elif n:
        part((0, n))
    return codes, scales


def e4m3_round(x: float) -> int:
    """Signed E4M3 byte of a real: nearest value, ties to the even code, 448 beyond."""
    return int(lib().oracle_e4m3_round(float(x)))


def project_ikeys(codes, scales, w_bits) -> np.ndarray:
    """Indexer keys projected from stored rows: codes [..., D/2], scales
    [..., D/16], w [D][DI] bf16 bits -> [..., DI] E4M3 bytes.
    "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
    index, select": the indexer's keys are a projection of the main cache entries."""
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    w = _np(w_bits, np.uint16)
    D = c.shape[-1] * 2
    DI = w.shape[1]
    assert w.shape[0] == D
    n = int(np.prod(c.shape[:-1])) if c.ndim > 1 else 1
    out = np.zeros(c.shape[:-1] + (DI,), np.uint8)
    lib().oracle_project_ikeys(_ptr(c), _ptr(s), n, D, _ptr(w), DI, _ptr(out))
    return out


# --------------------------------------------------------------------------
# MXFP4 indexer keys ("G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache
# entries, and why they're safe": 128 values x 4 bits + one 8-bit scale per 32
# values = 68 B).  A packed key row is its DI/2 code bytes then its DI/32
# scale bytes.
# --------------------------------------------------------------------------

def mx_exponent(amax: float) -> int:
    """Block exponent X = floor(log2 amax) - 2, clamped to [-8, 6] (-8 for 0)."""
    return int(lib().oracle_mx_exponent(float(amax)))


def mx_quantize(x) -> tuple:
    """Reals [..., DI] (float64) -> (codes [..., DI/2], scales [..., DI/32])."""
    a = _np(x, np.float64)
    DI = a.shape[-1]
    n = int(np.prod(a.shape[:-1])) if a.ndim > 1 else 1
    codes = np.zeros(a.shape[:-1] + (DI // 2,), np.uint8)
    scales = np.zeros(a.shape[:-1] + (DI // 32,), np.uint8)
    lib().oracle_mx_quantize(_ptr(a), n, DI, _ptr(codes), _ptr(scales))
    return codes, scales


def mx_quantize_bf16(x_bits) -> tuple:
    bits = _np(x_bits, np.uint16).astype(np.uint32) << 16
    return mx_quantize(bits.view(np.float32).astype(np.float64))


def mx_dequantize(codes, scales) -> np.ndarray:
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    DI = c.shape[-1] * 2
    n = int(np.prod(c.shape[:-1])) if c.ndim > 1 else 1
    out = np.zeros(c.shape[:-1] + (DI,), np.float64)
    lib().oracle_mx_dequantize(_ptr(c), _ptr(s), n, DI, _ptr(out))
    return out


def mx_pack(codes, scales) -> np.ndarray:
    return np.ascontiguousarray(np.concatenate([_np(codes, np.uint8), _np(scales, np.uint8)], axis=-1))


def mx_unpack(keys, DI: int) -> tuple:
    k = _np(keys, np.uint8)
    return np.ascontiguousarray(k[..., : DI // 2]), np.ascontiguousarray(k[..., DI // 2:])


def project_ikeys_mx(codes, scales, w_bits) -> np.ndarray:
    """Projected keys (as project_ikeys) in MXFP4: packed rows [..., DI/2 + DI/32]."""
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    w = _np(w_bits, np.uint16)
    D = c.shape[-1] * 2
    DI = w.shape[1]
    n = int(np.prod(c.shape[:-1])) if c.ndim > 1 else 1
    kc = np.zeros(c.shape[:-1] + (DI // 2,), np.uint8)
    ks = np.zeros(c.shape[:-1] + (DI // 32,), np.uint8)
    lib().oracle_project_ikeys_mx(_ptr(c), _ptr(s), n, D, _ptr(w), DI, _ptr(kc), _ptr(ks))
    return mx_pack(kc, ks)


def dequantize_rows(codes, scales) -> np.ndarray:
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    D = c.shape[-1] * 2
    n = int(np.prod(c.shape[:-1])) if c.ndim > 1 else 1
    out = np.zeros(c.shape[:-1] + (D,), np.float64)
    lib().oracle_dequantize_rows(_ptr(c), _ptr(s), n, D, _ptr(out))
    return out


class Cache:
    """Host copy of one global cache: rows [0, lengths[b]) of each sequence are valid.
    Indexer keys are E4M3 rows [DI] ("e4m3") or packed MXFP4 rows [DI/2 + DI/32] ("mxfp4")."""

    def __init__(self, B: int, capacity: int, D: int, DI: int, key_format: str = "e4m3"):
        self.B, self.capacity, self.D, self.DI = B, capacity, D, DI
        self.key_format = key_format
        self.codes = np.zeros((B, capacity, D // 2), np.uint8)
        self.scales = np.zeros((B, capacity, D // 16), np.uint8)
        kb = DI if key_format == "e4m3" else DI // 2 + DI // 32
        self.ikeys = np.zeros((B, capacity, kb), np.uint8)
        self.lengths = np.zeros(B, np.int64)

    def append(self, rows_bits, ikeys, threads: int = 1) -> None:
        """Quantise rows [B, n, D] and write them, with their ikeys [B, n, key bytes],
        at positions lengths[b] .. lengths[b]+n-1; then lengths += n."""
        rows = _np(rows_bits, np.uint16)
        ik = _np(ikeys, np.uint8)
        n = rows.shape[1]
        codes, scales = quantize_rows(rows, threads)
        for b in range(self.B):
            l0 = int(self.lengths[b])
            assert l0 + n <= self.capacity
            self.codes[b, l0:l0 + n] = codes[b]
            self.scales[b, l0:l0 + n] = scales[b]
            self.ikeys[b, l0:l0 + n] = ik[b]
            self.lengths[b] = l0 + n


# --------------------------------------------------------------------------
# next: persistent cache records ("G2C Brief", section "FP4 cache entries, and
# why they're safe", the derivation of the 890 bytes per token)
# --------------------------------------------------------------------------

def record_bytes(D: int, DI: int, key_format: str = "e4m3") -> int:
    """Bytes of one cache entry's record: D/2 + D/16 + the indexer entry's bytes."""
    return int(lib().oracle_record_bytes(D, DI, 1 if key_format == "mxfp4" else 0))


def bytes_per_token(records: Sequence[int], ms: Sequence[int]) -> float:
    """Bytes per token of the caches of several layers, layer i keeping one
    record of records[i] bytes per ms[i] tokens."""
    r = np.ascontiguousarray(records, np.int64)
    m = np.ascontiguousarray(ms, np.int32)
    return float(lib().oracle_bytes_per_token(_ptr(r), _ptr(m), len(r)))


def cache_spill(cache: "Cache", row0: int, n: int) -> np.ndarray:
    """Records of rows [row0, row0 + n) of every sequence: uint8 [B, n, record]
    (zeros for rows at or past the sequence's length)."""
    mx = 1 if cache.key_format == "mxfp4" else 0
    rb = record_bytes(cache.D, cache.DI, cache.key_format)
    out = np.zeros((cache.B, n, rb), np.uint8)
    lengths = np.ascontiguousarray(cache.lengths, np.int64)
    lib().oracle_cache_spill(_ptr(cache.codes), _ptr(cache.scales), _ptr(cache.ikeys), cache.B, cache.capacity,
                             cache.D, cache.DI, mx, _ptr(lengths), row0, n, _ptr(out))
    return out


def cache_reload(cache: "Cache", records) -> int:
    """Appends records [B, n, record] to every sequence (in place); returns the
    number of sequences left unchanged because they would pass capacity."""
    mx = 1 if cache.key_format == "mxfp4" else 0
    rec = _np(records, np.uint8)
    lengths = np.ascontiguousarray(cache.lengths, np.int64)
    skipped = lib().oracle_cache_reload(_ptr(cache.codes), _ptr(cache.scales), _ptr(cache.ikeys), cache.B,
                                        cache.capacity, cache.D, cache.DI, mx, _ptr(lengths), _ptr(rec),
                                        rec.shape[1])
    cache.lengths[:] = lengths
    return int(skipped)


def visible_length(length: int, P: int, p: int) -> int:
    """Causal visibility of query position p of P: the last P cached rows are the
    step's own positions, and position p sees rows [0, length - P + 1 + p)."""
    return int(length) - P + 1 + p


# --------------------------------------------------------------------------
# a2 / a4: indexer scores
# --------------------------------------------------------------------------

def index_scores(iq, w, ikeys_b, rows, threads: int = 1) -> np.ndarray:
    """Scores of candidate rows for one query: iq [HI, DI] E4M3, w [HI] fp32,
    ikeys_b [n_rows_total, DI], rows: int64 row ids -> fp32 [len(rows)].
    threads > 1 splits the candidate rows over threads."""
    q = _np(iq, np.uint8)
    ww = _np(w, np.float32)
    ik = _np(ikeys_b, np.uint8)
    r = np.ascontiguousarray(np.asarray(rows, np.int64))
    HI, DI = q.shape
    out = np.zeros(r.shape[0], np.float32)

    def part(c):
        a, b = c
        lib().oracle_index_score(_ptr(q), _ptr(ww), HI, DI, _ptr(ik), _ptr(r[a:b]), b - a, _ptr(out[a:b]))

    if threads > 1 and r.shape[0] > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, _chunks(r.shape[0], threads)))
    elif r.shape[0]:
        part((0, r.shape[0]))
    return out


def index_scores_mx(iq, w, keys_b, rows, threads: int = 1) -> np.ndarray:
    """index_scores with MXFP4 keys: keys_b [n_rows_total, DI/2 + DI/32] packed rows."""
    q = _np(iq, np.uint8)
    ww = _np(w, np.float32)
    HI, DI = q.shape
    kc, ks = mx_unpack(keys_b, DI)
    r = np.ascontiguousarray(np.asarray(rows, np.int64))
    out = np.zeros(r.shape[0], np.float32)

    def part(c):
        a, b = c
        lib().oracle_index_score_mx(_ptr(q), _ptr(ww), HI, DI, _ptr(kc), _ptr(ks), _ptr(r[a:b]), b - a,
                                    _ptr(out[a:b]))

    if threads > 1 and r.shape[0] > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, _chunks(r.shape[0], threads)))
    elif r.shape[0]:
        part((0, r.shape[0]))
    return out


def pool_rows(pool_blocks_ids, L_p: int):
    """Candidate rows of a block pool (block ids ascending, -1 = empty slot):
    returns (rows int64 [8*len(pool)], valid uint8) in pool order, member order."""
    pool = np.asarray(pool_blocks_ids, np.int64)
    rows = (pool[:, None] * POOL_BLOCK + np.arange(POOL_BLOCK)[None, :]).reshape(-1)
    valid = ((np.repeat(pool, POOL_BLOCK) >= 0) & (rows < L_p)).astype(np.uint8)
    rows = np.where(valid.astype(bool), rows, 0)
    return rows, valid


# --------------------------------------------------------------------------
# a3: selection
# --------------------------------------------------------------------------

def topk(scores, K: int, valid=None) -> np.ndarray:
    """Indices of the K largest scores (ties: lower index) in rank order, -1 padded."""
    s = _np(scores, np.float32)
    n = s.shape[0]
    out = np.zeros(K, np.int64)
    v = None if valid is None else np.ascontiguousarray(np.asarray(valid, np.uint8))
    lib().oracle_topk(_ptr(s), None if v is None else _ptr(v), n, K, _ptr(out))
    return out


def block_max(scores, block: int = POOL_BLOCK) -> np.ndarray:
    s = _np(scores, np.float32)
    n = s.shape[0]
    out = np.zeros((n + block - 1) // block, np.float32)
    if n:
        lib().oracle_block_max(_ptr(s), n, block, _ptr(out))
    return out


def build_pool(scores_full, n_keep: int) -> np.ndarray:
    """Hierarchical pool from one query's full scores: the n_keep blocks of 8
    with the best member score (ties: lower block id), returned as block ids in
    ascending order followed by -1 padding."""
    bs = block_max(scores_full)
    sel = topk(bs, n_keep)
    kept = np.sort(sel[sel >= 0])
    return np.concatenate([kept, -np.ones(n_keep - kept.shape[0], np.int64)])


# --------------------------------------------------------------------------
# a5 / a6: sparse attention
# --------------------------------------------------------------------------

def attend(q_bits, codes_b, scales_b, idx, scale: float):
    """q [H, D] bf16 bits; codes_b [rows, D/2]; scales_b [rows, D/16]; idx [K]
    -> (out fp32 [H, D], lse fp32 [H])."""
    q = _np(q_bits, np.uint16)
    c = _np(codes_b, np.uint8)
    s = _np(scales_b, np.uint8)
    ix = np.ascontiguousarray(np.asarray(idx, np.int64))
    H, D = q.shape
    out = np.zeros((H, D), np.float32)
    lse = np.zeros(H, np.float32)
    lib().oracle_attend(_ptr(q), H, D, float(scale), _ptr(c), _ptr(s), _ptr(ix), ix.shape[0],
                        _ptr(out), _ptr(lse))
    return out, lse


def swa_window(n_swa: int, P: int, p: int, window: int):
    """Rows [lo, hi) of a sequence's local cache that position p attends to:
    the `window` most recent tokens up to and including its own, whose row is
    n_swa - P + p (the step's P positions are the last P local rows).
    "G2C Brief - DeepSeek V4.1-Flash", section "Two attention paths in every
    layer": exact sliding-window attention over the most recent 128 tokens."""
    own = n_swa - P + p
    return max(0, own - window + 1), own + 1


def attend_swa(q_bits, codes_b, scales_b, idx, swa_b, lo: int, hi: int, scale: float):
    """Joint softmax over the selected FP4 rows and the FP8 E4M3 window rows
    swa_b[lo:hi] (one shared latent per token, K = V).  q [H, D] bf16 bits;
    swa_b [n_swa, D] E4M3 bytes -> (out fp32 [H, D], lse fp32 [H])."""
    q = _np(q_bits, np.uint16)
    c = _np(codes_b, np.uint8)
    s = _np(scales_b, np.uint8)
    w = _np(swa_b, np.uint8)
    ix = np.ascontiguousarray(np.asarray(idx, np.int64))
    H, D = q.shape
    out = np.zeros((H, D), np.float32)
    lse = np.zeros(H, np.float32)
    lib().oracle_attend_swa(_ptr(q), H, D, float(scale), _ptr(c), _ptr(s), _ptr(ix), ix.shape[0], _ptr(w),
                            int(lo), int(hi), _ptr(out), _ptr(lse))
    return out, lse


# --------------------------------------------------------------------------
# a7: one query through one layer, and the mode chain
# --------------------------------------------------------------------------

def unit_layer(cache: Cache, b: int, p: int, P: int, mode: int, q, iq, w, K: int, scale: float,
               prev_idx=None, pool_in=None, pool_keep: int = 0, threads: int = 1,
               swa=None) -> Dict[str, np.ndarray]:
    """One (sequence b, position p) through one CSA2 layer.

    Full    : score every visible row, keep the top K (and, with pool_keep > 0,
              the best pool_keep blocks of 8 as the hierarchical pool).
    Reindex : score the visible rows again with this layer's own indexer
              query, or only the pool's rows when pool_in is given; fresh top K.
    Reuse   : take prev_idx unchanged.
    Then attend over the selected rows with this layer's own query; with
    swa = (rows_b [n, D] E4M3 bytes of this sequence, window), jointly with the
    local window of this position (attend_swa).
    """
    L_p = visible_length(cache.lengths[b], P, p)
    res: Dict[str, np.ndarray] = {}
    if mode == REUSE:
        idx = np.asarray(prev_idx, np.int64)
    elif mode == REINDEX and pool_in is not None:
        rows, valid = pool_rows(pool_in, L_p)
        sc = (index_scores_mx if cache.key_format == "mxfp4" else index_scores)(iq, w, cache.ikeys[b], rows, threads)
        sel = topk(sc, K, valid)
        idx = np.where(sel >= 0, rows[np.maximum(sel, 0)], -1)
        res["scores"], res["rows"], res["valid"] = sc, rows, valid
    else:
        rows = np.arange(L_p, dtype=np.int64)
        sc = (index_scores_mx if cache.key_format == "mxfp4" else index_scores)(iq, w, cache.ikeys[b], rows, threads)
        idx = topk(sc, K)
        res["scores"] = sc
        if mode == FULL and pool_keep:
            res["pool"] = build_pool(sc, pool_keep)
    if swa is None:
        out, lse = attend(q, cache.codes[b], cache.scales[b], idx, scale)
    else:
        rows_b, window = swa
        lo, hi = swa_window(rows_b.shape[0], P, p, window)
        out, lse = attend_swa(q, cache.codes[b], cache.scales[b], idx, rows_b, lo, hi, scale)
    res.update(idx=idx, out=out, lse=lse)
    return res


def run_layer(cache: Cache, mode: int, inputs: Dict, K: int, scale: float, P: int = 1,
              prev_idx=None, pool_in=None, pool_keep: int = 0,
              units: Optional[Sequence] = None, threads: int = 1, score_threads: int = 1,
              swa=None) -> Dict:
    """One layer for every (b, p) unit (or the listed units).  inputs holds
    q [B,P,H,D] bf16 bits, iq [B,P,HI,DI], w [B,P,HI]; swa = (rows [B, n, D]
    E4M3 bytes, window) or None.  Returns per-unit dicts."""
    q = _np(inputs["q"], np.uint16)
    iq = _np(inputs["iq"], np.uint8)
    w = _np(inputs["w"], np.float32)
    if units is None:
        units = [(b, p) for b in range(cache.B) for p in range(P)]

    def one(u):
        b, p = u
        return u, unit_layer(cache, b, p, P, mode, q[b, p], iq[b, p], w[b, p], K, scale,
                             None if prev_idx is None else prev_idx[u],
                             None if pool_in is None else pool_in[u], pool_keep, score_threads,
                             None if swa is None else (swa[0][b], swa[1]))

    if threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            return dict(ex.map(one, units))
    return dict(map(one, units))


def run_chain(cache: Cache, modes: Sequence[int], layer_inputs: Sequence[Dict], K: int, scale: float,
              P: int = 1, pool_keep: int = 0, units=None, threads: int = 1, score_threads: int = 1,
              swa=None):
    """A chain of layers sharing one cache.  Reuse takes the nearest preceding
    Full/Reindex selection; Reindex uses the pool of the first Full layer when
    pool_keep > 0; swa = (rows [B, n, D], window) joins every layer's attention
    to the local window.  Returns a list of per-layer results."""
    results, prev, pool = [], None, None
    for li, mode in enumerate(modes):
        r = run_layer(cache, mode, layer_inputs[li], K, scale, P,
                      prev_idx=prev if mode == REUSE else None,
                      pool_in=pool if mode == REINDEX else None,
                      pool_keep=pool_keep if (mode == FULL and pool is None) else 0,
                      units=units, threads=threads, score_threads=score_threads, swa=swa)
        if mode != REUSE:
            prev = {u: v["idx"] for u, v in r.items()}
        if mode == FULL and pool is None and pool_keep:
            pool = {u: v["pool"] for u, v in r.items()}
        results.append(r)
    return results
