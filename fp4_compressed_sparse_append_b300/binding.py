"""Thin ctypes binding of libcsa (the C ABI declared in include/csa.h).

Every function here only marshals torch tensors (device memory owned by
torch) and the current CUDA stream into the C calls of the same name; every
step of the computation runs in the library's CUDA kernels.  There is no CPU
path: if libcsa.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

CSA_FULL, CSA_REINDEX, CSA_REUSE = 0, 1, 2
CSA_POOL_BLOCK = 8
CSA_NOALLOC_SCRATCH_BYTES = 17 << 20
CSA_DEV_BAD_INDEX, CSA_DEV_CAPACITY, CSA_DEV_TIMEOUT = 0x1, 0x2, 0x4

EXPORTS = (
    "csa_quantize_append", "csa_quantize_append_project", "csa_index_score", "csa_topk", "csa_topk_workspace_size",
    "csa_pool_topk", "csa_pool_topk_workspace_size", "csa_select_pairs", "csa_topk_pairs", "csa_ids_window", "csa_lse_merge", "csa_sparse_attend",
    "csa_sparse_attend_noalloc", "csa_sparse_attend_swa", "csa_attend_swa_workspace_size",
    "csa_attend_workspace_size", "csa_layer_step", "csa_layer_workspace_size",
    "csa_device_status", "csa_kernel_launches", "csa_status_string",
    "csa_cache_record_bytes", "csa_cache_spill", "csa_cache_reload",
)


class CsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))
        self.status = status


CSA_IKEY_E4M3, CSA_IKEY_MXFP4 = 0, 1


class csa_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("capacity", ctypes.c_int32), ("d_latent", ctypes.c_int32),
                ("d_index", ctypes.c_int32), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("ikeys", ctypes.c_void_p), ("lengths", ctypes.c_void_p), ("ikey_format", ctypes.c_int32),
                ("iscales", ctypes.c_void_p)]


class csa_swa(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_void_p), ("lengths", ctypes.c_void_p), ("n", ctypes.c_int32),
                ("window", ctypes.c_int32)]


class csa_layer_args(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("P", ctypes.c_int32), ("H", ctypes.c_int32), ("HI", ctypes.c_int32),
                ("K", ctypes.c_int32), ("scale", ctypes.c_float), ("q", ctypes.c_void_p),
                ("iq", ctypes.c_void_p), ("w", ctypes.c_void_p), ("rows_new", ctypes.c_void_p),
                ("ikeys_new", ctypes.c_void_p), ("n_new", ctypes.c_int32), ("pool_blocks", ctypes.c_int32),
                ("pool_in", ctypes.c_void_p), ("pool_out", ctypes.c_void_p), ("idx", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("swa", ctypes.c_void_p), ("w_ik", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libcsa.so (built by fp4_compressed_sparse_append_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libcsa.so is not built (run __graft_entry__.build()); "
                               "there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        V, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        C = ctypes.POINTER(csa_cache)
        L.csa_quantize_append.argtypes = [C, V, V, I32, V]
        L.csa_quantize_append_project.argtypes = [C, V, V, I32, V]
        L.csa_index_score.argtypes = [C, I32, I32, V, V, V, I32, V, I64, V, I64, V]
        L.csa_topk.argtypes = [C, I32, V, I64, V, I32, I32, V, I32, V, V, I64, V, SZ, V]
        L.csa_topk_workspace_size.argtypes = [C, I32, I32, I32, I32, ctypes.POINTER(SZ)]
        L.csa_pool_topk.argtypes = [C, I32, I32, V, V, V, I32, I32, V, V, SZ, V]
        L.csa_pool_topk_workspace_size.argtypes = [C, I32, I32, ctypes.POINTER(SZ)]
        L.csa_select_pairs.argtypes = [C, V, I64, V, I32, I32, I32, V, V, V]
        L.csa_topk_pairs.argtypes = [I32, I32, V, V, I32, V, V]
        L.csa_ids_window.argtypes = [V, I64, I32, I32, V, V]
        L.csa_lse_merge.argtypes = [I32, I32, I32, I32, V, V, V, V, V]
        L.csa_sparse_attend.argtypes = [C, I32, I32, V, ctypes.c_float, V, I32, V, V, V, SZ, V]
        L.csa_sparse_attend_noalloc.argtypes = [C, I32, I32, V, ctypes.c_float, V, I32, V, V, V]
        L.csa_attend_workspace_size.argtypes = [C, I32, I32, I32, ctypes.POINTER(SZ)]
        S = ctypes.POINTER(csa_swa)
        L.csa_sparse_attend_swa.argtypes = [C, I32, I32, V, ctypes.c_float, V, I32, S, V, V, V, SZ, V]
        L.csa_attend_swa_workspace_size.argtypes = [C, I32, I32, I32, S, ctypes.POINTER(SZ)]
        L.csa_layer_step.argtypes = [C, ctypes.POINTER(csa_layer_args), V]
        L.csa_layer_workspace_size.argtypes = [C, ctypes.POINTER(csa_layer_args), ctypes.POINTER(SZ)]
        L.csa_device_status.argtypes = [ctypes.POINTER(I32), I32, V]
        L.csa_kernel_launches.argtypes = []
        L.csa_kernel_launches.restype = ctypes.c_uint64
        L.csa_status_string.argtypes = [ctypes.c_int]
        L.csa_status_string.restype = ctypes.c_char_p
        L.csa_cache_record_bytes.argtypes = [C]
        L.csa_cache_record_bytes.restype = SZ
        L.csa_cache_spill.argtypes = [C, I32, I32, V, V]
        L.csa_cache_reload.argtypes = [C, V, I32, V]
        for name in EXPORTS:
            if name not in ("csa_status_string", "csa_kernel_launches", "csa_cache_record_bytes"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().csa_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise CsaError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _need(t: Optional[torch.Tensor], nbytes: int, name: str) -> None:
    """The C ABI sees only a pointer: a tensor smaller than the bytes the call
    reads or writes would let a kernel run past it, so it is refused here."""
    if t is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError("%s holds %d bytes; the call touches %d" % (name, t.numel() * t.element_size(), nbytes))


def _lead(t: torch.Tensor, name: str, batch: int, last: Optional[int] = None) -> None:
    """Outputs are allocated from this tensor's shape: its batch (and last) dims
    must be the cache's."""
    if t.shape[0] != batch or (last is not None and t.shape[-1] != last):
        raise ValueError("%s has shape %s; expected [%d, ...%s]" % (name, tuple(t.shape), batch,
                                                                    "" if last is None else ", %d" % last))


def _key_row_bytes(cache: "Cache") -> int:
    """Bytes of one appended indexer key row (E4M3: DI; MXFP4: DI/2 codes + DI/32 scales)."""
    return cache.d_index // 2 + cache.d_index // 32 if cache.key_format == "mxfp4" else cache.d_index


def _need_attend(cache: "Cache", P: int, H: int, K: int, q, idx, out, lse, swa=None) -> None:
    Bc, D = cache.batch, cache.d_latent
    _need(q, Bc * P * H * D * 2, "q")
    _need(idx, Bc * P * K * 4, "idx")
    _need(out, Bc * P * H * D * 4, "out")
    _need(lse, Bc * P * H * 4, "lse")
    if swa is not None:
        _need(swa.rows, Bc * swa.rows.shape[1] * D, "swa rows")
        _need(swa.lengths, Bc * 4, "swa lengths")


def _ptr_dev_or_pinned(t: torch.Tensor):
    """Device tensors, or pinned host tensors (which the device addresses directly)."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("expected a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Cache:
    """A global FP4 cache in device memory (torch tensors), laid out as csa_cache says.

    codes [B, cap, D/2] u8, scales [B, cap, D/16] u8, lengths [B] i32; indexer keys
    ikeys [B, cap, DI] u8 (E4M3), or for key_format="mxfp4" ikeys [B, cap, DI/2]
    (E2M1 codes) and iscales [B, cap, DI/32] (UE8M0 block scales).
    """

    def __init__(self, batch: int, capacity: int, d_latent: int, d_index: int, device="cuda",
                 key_format: str = "e4m3"):
        self.batch, self.capacity, self.d_latent, self.d_index = batch, capacity, d_latent, d_index
        self.key_format = key_format
        mx = key_format == "mxfp4"
        dev = torch.device(device)
        self.codes = torch.zeros((batch, capacity, d_latent // 2), dtype=torch.uint8, device=dev)
        self.scales = torch.zeros((batch, capacity, d_latent // 16), dtype=torch.uint8, device=dev)
        self.ikeys = torch.zeros((batch, capacity, d_index // 2 if mx else d_index), dtype=torch.uint8, device=dev)
        self.iscales = torch.zeros((batch, capacity, d_index // 32), dtype=torch.uint8, device=dev) if mx else None
        self.lengths = torch.zeros((batch,), dtype=torch.int32, device=dev)
        self._struct = csa_cache(batch, capacity, d_latent, d_index, self.codes.data_ptr(),
                                 self.scales.data_ptr(), self.ikeys.data_ptr(), self.lengths.data_ptr(),
                                 CSA_IKEY_MXFP4 if mx else CSA_IKEY_E4M3,
                                 self.iscales.data_ptr() if mx else None)

    def packed_keys(self) -> torch.Tensor:
        """MXFP4 keys as packed rows [B, cap, DI/2 + DI/32] (codes then scales)."""
        return torch.cat([self.ikeys, self.iscales], dim=-1)

    @property
    def ref(self):
        return ctypes.byref(self._struct)

    @property
    def device(self):
        return self.codes.device


# ---------------------------------------------------------------------------
# The calls of include/csa.h
# ---------------------------------------------------------------------------

def csa_quantize_append(cache: Cache, rows: torch.Tensor, ikeys_new: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """rows: [B, n, D] bf16 (or its int16 bits); ikeys_new: [B, n, DI] uint8 or None."""
    n = rows.shape[1]
    _need(rows, cache.batch * n * cache.d_latent * 2, "rows")
    _need(ikeys_new, cache.batch * n * _key_row_bytes(cache), "ikeys_new")
    _check(lib().csa_quantize_append(cache.ref, _ptr(rows), _ptr(ikeys_new), n, _stream(stream)),
           "csa_quantize_append")


def csa_quantize_append_project(cache: Cache, rows: torch.Tensor, w_ik: torch.Tensor, stream=None) -> None:
    """rows: [B, n, D] bf16 bits; w_ik: [D, DI] bf16 bits.  The appended rows'
    indexer keys are projected from their stored FP4 entries."""
    n = rows.shape[1]
    _need(rows, cache.batch * n * cache.d_latent * 2, "rows")
    _need(w_ik, cache.d_latent * cache.d_index * 2, "w_ik")
    _check(lib().csa_quantize_append_project(cache.ref, _ptr(rows), _ptr(w_ik), n, _stream(stream)),
           "csa_quantize_append_project")


def csa_cache_record_bytes(cache: Cache) -> int:
    """Bytes of one persistent record (main entry codes and scales, then the indexer entry)."""
    return int(lib().csa_cache_record_bytes(cache.ref))


def csa_cache_spill(cache: Cache, row0: int, n: int, records: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Records of rows [row0, row0 + n) of every sequence -> uint8 [B, n, record]
    (device memory, or the given tensor: device or pinned host memory)."""
    if records is None:
        records = torch.empty((cache.batch, n, csa_cache_record_bytes(cache)), dtype=torch.uint8,
                              device=cache.device)
    _need(records, cache.batch * n * csa_cache_record_bytes(cache), "records")
    _check(lib().csa_cache_spill(cache.ref, row0, n, _ptr_dev_or_pinned(records), _stream(stream)),
           "csa_cache_spill")
    return records


def csa_cache_reload(cache: Cache, records: torch.Tensor, stream=None) -> None:
    """Appends records [B, n, record] (device or pinned host memory) to every sequence."""
    _need(records, cache.batch * records.shape[1] * csa_cache_record_bytes(cache), "records")
    _check(lib().csa_cache_reload(cache.ref, _ptr_dev_or_pinned(records), records.shape[1], _stream(stream)),
           "csa_cache_reload")


def block_max_buffer(cache: Cache, P: int) -> torch.Tensor:
    """An empty [B, P, ldb] fp32 buffer for csa_index_score's block maxima
    (ldb = ceil(capacity / 8) rounded up to 4)."""
    ldb = ((cache.capacity + CSA_POOL_BLOCK - 1) // CSA_POOL_BLOCK + 3) // 4 * 4
    return torch.empty((cache.batch, P, ldb), dtype=torch.float32, device=cache.device)


def csa_index_score(cache: Cache, iq: torch.Tensor, w: torch.Tensor, pool: Optional[torch.Tensor] = None,
                    scores: Optional[torch.Tensor] = None, block_max: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """iq [B, P, HI, DI] uint8, w [B, P, HI] fp32, pool [B, P, nblk] int32 or None
    -> scores [B, P, ld] fp32 (ld = capacity rounded up to 4, or 8*nblk).
    block_max [B, P, ldb] fp32 (block_max_buffer; full scans only) also
    receives each 8-row block's best visible score."""
    B, P, HI, _ = iq.shape
    _lead(iq, "iq", cache.batch, cache.d_index)
    nblk = pool.shape[-1] if pool is not None else 0
    n = nblk * CSA_POOL_BLOCK if pool is not None else cache.capacity
    if scores is None:
        scores = torch.empty((B, P, (n + 3) // 4 * 4), dtype=torch.float32, device=cache.device)
    Bc = cache.batch
    _need(iq, Bc * P * HI * cache.d_index, "iq")
    _need(w, Bc * P * HI * 4, "w")
    _need(pool, Bc * P * nblk * 4, "pool")
    _need(scores, Bc * P * scores.shape[-1] * 4, "scores")
    ldb = block_max.shape[-1] if block_max is not None else 0
    _need(block_max, Bc * P * ldb * 4, "block_max")
    _check(lib().csa_index_score(cache.ref, P, HI, _ptr(iq), _ptr(w), _ptr(pool), nblk, _ptr(scores),
                                 scores.shape[-1], _ptr(block_max), ldb, _stream(stream)), "csa_index_score")
    return scores


def topk_workspace_size(cache: Cache, P: int, K: int, pool_blocks: int = 0, pool_keep: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().csa_topk_workspace_size(cache.ref, P, pool_blocks, K, pool_keep, ctypes.byref(n)),
           "csa_topk_workspace_size")
    return n.value


def csa_topk(cache: Cache, scores: torch.Tensor, K: int, pool: Optional[torch.Tensor] = None,
             pool_keep: int = 0, block_max: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """scores [B, P, ld] -> (idx [B, P, K] int32, pool_out [B, P, pool_keep] int32 or None).
    block_max: the block maxima csa_index_score wrote beside these scores
    (with pool_keep > 0), from which the pool is then selected."""
    B, P, ld = scores.shape
    _lead(scores, "scores", cache.batch)
    nblk = pool.shape[-1] if pool is not None else 0
    _need(scores, cache.batch * P * ld * 4, "scores")
    _need(pool, cache.batch * P * nblk * 4, "pool")
    ldb = block_max.shape[-1] if block_max is not None else 0
    _need(block_max, cache.batch * P * ldb * 4, "block_max")
    idx = torch.empty((B, P, K), dtype=torch.int32, device=cache.device)
    pool_out = torch.empty((B, P, pool_keep), dtype=torch.int32, device=cache.device) if pool_keep else None
    if workspace is None:
        n = topk_workspace_size(cache, P, K, nblk, pool_keep)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
    _check(lib().csa_topk(cache.ref, P, _ptr(scores), ld, _ptr(pool), nblk, K, _ptr(idx), pool_keep,
                          _ptr(pool_out), _ptr(block_max), ldb, _ptr(workspace), workspace.numel(),
                          _stream(stream)), "csa_topk")
    return idx, pool_out


def pool_topk_workspace_size(cache: Cache, P: int, pool_blocks: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().csa_pool_topk_workspace_size(cache.ref, P, pool_blocks, ctypes.byref(n)),
           "csa_pool_topk_workspace_size")
    return n.value


def csa_pool_topk(cache: Cache, iq: torch.Tensor, w: torch.Tensor, pool: torch.Tensor, K: int,
                  idx: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Reindex over a pool in one call: iq [B, P, HI, DI] uint8, w [B, P, HI]
    fp32, pool [B, P, nblk] int32 -> idx [B, P, K] int32 (the top K of the
    pool's rows, ascending, -1 padded).  workspace (pool_topk_workspace_size
    bytes) selects the spread form, None the cluster form."""
    B, P, HI, _ = iq.shape
    _lead(iq, "iq", cache.batch, cache.d_index)
    nblk = pool.shape[-1]
    Bc = cache.batch
    _need(iq, Bc * P * HI * cache.d_index, "iq")
    _need(w, Bc * P * HI * 4, "w")
    _need(pool, Bc * P * nblk * 4, "pool")
    if idx is None:
        idx = torch.empty((B, P, K), dtype=torch.int32, device=cache.device)
    _need(idx, Bc * P * K * 4, "idx")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(lib().csa_pool_topk(cache.ref, P, HI, _ptr(iq), _ptr(w), _ptr(pool), nblk, K, _ptr(idx), ws_ptr, ws_bytes,
                               _stream(stream)), "csa_pool_topk")
    return idx


def csa_select_pairs(cache: Cache, scores: torch.Tensor, idx: torch.Tensor, block: int, id_offset: int,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """scores [B, 1, ld] fp32 of the cache's rows, idx [B, 1, n] int32 local ids
    (rows, or blocks of 8 rows with block=8) -> (pair_scores [B, 1, n] fp32,
    pair_ids [B, 1, n] int32 = id + id_offset, -1 for empty slots)."""
    Bc, n = cache.batch, idx.shape[-1]
    _need(scores, Bc * scores.shape[-1] * 4, "scores")
    _need(idx, Bc * n * 4, "idx")
    ps = torch.empty((Bc, 1, n), dtype=torch.float32, device=cache.device)
    pi = torch.empty((Bc, 1, n), dtype=torch.int32, device=cache.device)
    _check(lib().csa_select_pairs(cache.ref, _ptr(scores), scores.shape[-1], _ptr(idx), n, block, id_offset,
                                  _ptr(ps), _ptr(pi), _stream(stream)), "csa_select_pairs")
    return ps, pi


def csa_topk_pairs(pair_scores: torch.Tensor, pair_ids: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """pair_scores / pair_ids [rows, n] -> idx [rows, K] int32 (the ids of the K
    best pairs, in pair order, -1 padded)."""
    rows, n = pair_scores.shape[0], pair_scores.shape[-1]
    ps, pi = pair_scores.reshape(rows, n).contiguous(), pair_ids.reshape(rows, n).contiguous()
    idx = torch.empty((rows, K), dtype=torch.int32, device=ps.device)
    _check(lib().csa_topk_pairs(rows, n, _ptr(ps), _ptr(pi), K, _ptr(idx), _stream(stream)), "csa_topk_pairs")
    return idx


def csa_ids_window(ids: torch.Tensor, lo: int, hi: int, stream=None) -> torch.Tensor:
    """ids - lo where lo <= ids < hi, else -1 (same shape, int32)."""
    ids = ids.contiguous()
    out = torch.empty_like(ids)
    _check(lib().csa_ids_window(_ptr(ids), ids.numel(), lo, hi, _ptr(out), _stream(stream)), "csa_ids_window")
    return out


def csa_lse_merge(outs: torch.Tensor, lses: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """outs [parts, units..., H, D] fp32, lses [parts, units..., H] fp32 ->
    (out [units..., H, D], lse [units..., H]): the log-sum-exp merge."""
    parts, H, D = outs.shape[0], outs.shape[-2], outs.shape[-1]
    units = outs[0].numel() // (H * D)
    o, l = outs.contiguous(), lses.contiguous()
    out = torch.empty(outs.shape[1:], dtype=torch.float32, device=outs.device)
    lse = torch.empty(lses.shape[1:], dtype=torch.float32, device=outs.device)
    _check(lib().csa_lse_merge(parts, units, H, D, _ptr(o), _ptr(l), _ptr(out), _ptr(lse), _stream(stream)),
           "csa_lse_merge")
    return out, lse


def attend_workspace_size(cache: Cache, P: int, H: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().csa_attend_workspace_size(cache.ref, P, H, K, ctypes.byref(n)), "csa_attend_workspace_size")
    return n.value


def csa_sparse_attend(cache: Cache, q: torch.Tensor, idx: torch.Tensor, scale: float,
                      workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q [B, P, H, D] bf16 bits, idx [B, P, K] int32 -> (out [B, P, H, D] fp32, lse [B, P, H] fp32)."""
    B, P, H, D = q.shape
    _lead(q, "q", cache.batch, cache.d_latent)
    K = idx.shape[-1]
    _need_attend(cache, P, H, K, q, idx, out, lse)
    if workspace is None:
        workspace = torch.empty(attend_workspace_size(cache, P, H, K), dtype=torch.uint8, device=cache.device)
    if out is None:
        out = torch.empty((B, P, H, D), dtype=torch.float32, device=cache.device)
    if lse is None:
        lse = torch.empty((B, P, H), dtype=torch.float32, device=cache.device)
    _check(lib().csa_sparse_attend(cache.ref, P, H, _ptr(q), scale, _ptr(idx), K, _ptr(out), _ptr(lse),
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "csa_sparse_attend")
    return out, lse


def csa_sparse_attend_noalloc(cache: Cache, q: torch.Tensor, idx: torch.Tensor, scale: float,
                              out: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None) -> None:
    """Sparse attention into caller-provided out/lse, with the library's own
    fixed device scratch (no workspace argument; the call allocates nothing)."""
    B, P, H, D = q.shape
    _lead(q, "q", cache.batch, cache.d_latent)
    K = idx.shape[-1]
    _need_attend(cache, P, H, K, q, idx, out, lse)
    _check(lib().csa_sparse_attend_noalloc(cache.ref, P, H, _ptr(q), scale, _ptr(idx), K, _ptr(out), _ptr(lse),
                                           _stream(stream)), "csa_sparse_attend_noalloc")


class Swa:
    """The local window of csa_swa: rows [B, n, D] FP8 E4M3 bytes (uint8) and
    lengths [B] int32 (local rows per sequence) or None (n for every sequence)."""

    def __init__(self, rows: torch.Tensor, window: int, lengths: Optional[torch.Tensor] = None):
        self.rows, self.lengths, self.window = rows, lengths, window
        self._struct = csa_swa(_ptr(rows), _ptr(lengths), rows.shape[1], window)

    @property
    def ref(self):
        return ctypes.byref(self._struct)


def attend_swa_workspace_size(cache: Cache, P: int, H: int, K: int, swa: Optional[Swa]) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().csa_attend_swa_workspace_size(cache.ref, P, H, K, swa.ref if swa is not None else None,
                                               ctypes.byref(n)), "csa_attend_swa_workspace_size")
    return n.value


def csa_sparse_attend_swa(cache: Cache, q: torch.Tensor, idx: torch.Tensor, scale: float, swa: Optional[Swa],
                          workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Joint softmax over the selected rows and the local window -> (out [B, P, H, D], lse [B, P, H])."""
    B, P, H, D = q.shape
    _lead(q, "q", cache.batch, cache.d_latent)
    K = idx.shape[-1]
    _need_attend(cache, P, H, K, q, idx, out, lse, swa)
    if workspace is None:
        workspace = torch.empty(max(attend_swa_workspace_size(cache, P, H, K, swa), 16), dtype=torch.uint8,
                                device=cache.device)
    if out is None:
        out = torch.empty((B, P, H, D), dtype=torch.float32, device=cache.device)
    if lse is None:
        lse = torch.empty((B, P, H), dtype=torch.float32, device=cache.device)
    _check(lib().csa_sparse_attend_swa(cache.ref, P, H, _ptr(q), scale, _ptr(idx), K,
                                       swa.ref if swa is not None else None, _ptr(out), _ptr(lse),
                                       _ptr(workspace), workspace.numel(), _stream(stream)), "csa_sparse_attend_swa")
    return out, lse


class LayerArgs:
    """Owns the tensors of one csa_layer_step call and its csa_layer_args struct."""

    def __init__(self, cache: Cache, mode: int, q, K: int, scale: float, iq=None, w=None, idx=None,
                 rows_new=None, ikeys_new=None, pool_in=None, pool_blocks: int = 0, make_pool: bool = False,
                 swa: Optional[Swa] = None, w_ik=None, out=None, lse=None):
        B, P, H, D = q.shape
        _lead(q, "q", cache.batch, cache.d_latent)
        dev = cache.device
        self.tensors = dict(q=q, iq=iq, w=w, rows_new=rows_new, ikeys_new=ikeys_new, pool_in=pool_in)
        self.idx = idx if idx is not None else torch.empty((B, P, K), dtype=torch.int32, device=dev)
        self.out = out if out is not None else torch.empty((B, P, H, D), dtype=torch.float32, device=dev)
        self.lse = lse if lse is not None else torch.empty((B, P, H), dtype=torch.float32, device=dev)
        _need(self.out, B * P * H * D * 4, "out")
        _need(self.lse, B * P * H * 4, "lse")
        self.pool_out = (torch.empty((B, P, pool_blocks), dtype=torch.int32, device=dev)
                         if make_pool else None)
        HI = iq.shape[2] if iq is not None else 0
        n_new = rows_new.shape[1] if rows_new is not None else 0
        Bc = cache.batch
        _need_attend(cache, P, H, K, q, idx, None, None, swa)
        _need(iq, Bc * P * HI * cache.d_index, "iq")
        _need(w, Bc * P * HI * 4, "w")
        _need(rows_new, Bc * n_new * cache.d_latent * 2, "rows_new")
        _need(ikeys_new, Bc * n_new * _key_row_bytes(cache), "ikeys_new")
        _need(pool_in, Bc * P * pool_blocks * 4, "pool_in")
        _need(w_ik, cache.d_latent * cache.d_index * 2, "w_ik")
        self.struct = csa_layer_args(mode, P, H, HI, K, scale, _ptr(q), _ptr(iq), _ptr(w), _ptr(rows_new),
                                     _ptr(ikeys_new), n_new, pool_blocks, _ptr(pool_in), _ptr(self.pool_out),
                                     _ptr(self.idx), _ptr(self.out), _ptr(self.lse), None, 0,
                                     ctypes.addressof(swa._struct) if swa is not None else None, _ptr(w_ik))
        self.swa = swa
        self.tensors["w_ik"] = w_ik
        n = ctypes.c_size_t(0)
        _check(lib().csa_layer_workspace_size(cache.ref, ctypes.byref(self.struct), ctypes.byref(n)),
               "csa_layer_workspace_size")
        self.workspace = torch.empty(max(n.value, 16), dtype=torch.uint8, device=dev)
        self.struct.workspace = self.workspace.data_ptr()
        self.struct.workspace_bytes = self.workspace.numel()


def csa_layer_step(cache: Cache, args: LayerArgs, stream=None) -> LayerArgs:
    _check(lib().csa_layer_step(cache.ref, ctypes.byref(args.struct), _stream(stream)), "csa_layer_step")
    return args


def csa_kernel_launches() -> int:
    """Kernels launched by the library so far in this process (host counter)."""
    return int(lib().csa_kernel_launches())


def csa_device_status(clear: bool = True, stream=None) -> int:
    """Waits for the stream and returns the device status bits (0 = no fault)."""
    bits = ctypes.c_int32(0)
    st = lib().csa_device_status(ctypes.byref(bits), 1 if clear else 0, _stream(stream))
    if st not in (0, 4):
        _check(st, "csa_device_status")
    return bits.value
