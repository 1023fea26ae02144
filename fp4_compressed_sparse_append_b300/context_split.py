"""The context split of one long sequence over several devices.

"G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
index, select": every cached entry is scored, the query keeps the best and
attends to only those.  When one sequence's cache is too long for one device
(a 1M-token context), its rows are split into contiguous slices, one per
device (rank), and a layer runs as:

1. each rank scores its own slice and keeps its local top K, as (score,
   global row id) pairs (csa_index_score, csa_topk, csa_select_pairs);
2. exchange 1: every rank gathers every rank's K pairs;
3. every rank takes the global top K among the G*K pairs (csa_topk_pairs).
   This is exact: a row of the global top K is in its own slice's top K,
   since the same order (score, then lower id) decides both;
4. each rank attends over the selected rows that lie in its slice
   (csa_ids_window, csa_sparse_attend), which is the softmax over those rows;
5. exchange 2: every rank gathers every rank's (out, lse) and merges them by
   log-sum-exp (csa_lse_merge), which is the softmax over all selected rows.

Reuse layers skip 1-3 and attend over the previous selection.  One query
position per sequence (decode).  Slice boundaries are multiples of 8 rows.

The device steps go through ``ops`` (by default the library's C ABI, on the
rank's device); the exchanges through ``gather``, a callable that returns
every rank's copy of a tensor in rank order (``torch_gather`` for a
``torch.distributed`` group).  The phase functions let one process run several
ranks' steps in turn.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import binding as B

Tensor = torch.Tensor


def slice_rows(L: int, G: int, g: int) -> Tuple[int, int]:
    """Rows [lo, hi) of rank g of G for a sequence of L rows: contiguous,
    boundaries at multiples of 8 (a pool block never straddles two ranks)."""
    blocks = (L + 7) // 8
    lo = min(L, (blocks * g // G) * 8)
    hi = min(L, (blocks * (g + 1) // G) * 8)
    return lo, hi


@dataclasses.dataclass
class Part:
    """One rank's slice: its own cache of rows [row0, row0 + rows) of every
    sequence (row r of the cache is global row row0 + r)."""
    cache: object
    row0: int
    rows: int


class CudaOps:
    """The device steps, through the library's C ABI."""

    @staticmethod
    def index_score(cache, iq, w):
        return B.csa_index_score(cache, iq, w)

    @staticmethod
    def topk(cache, scores, K):
        return B.csa_topk(cache, scores, K)[0]

    @staticmethod
    def select_pairs(cache, scores, idx, id_offset):
        return B.csa_select_pairs(cache, scores, idx, 1, id_offset)

    @staticmethod
    def topk_pairs(pair_scores, pair_ids, K):
        return B.csa_topk_pairs(pair_scores, pair_ids, K)

    @staticmethod
    def ids_window(ids, lo, hi):
        return B.csa_ids_window(ids, lo, hi)

    @staticmethod
    def attend(cache, q, idx, scale):
        return B.csa_sparse_attend(cache, q, idx, scale)

    @staticmethod
    def lse_merge(outs, lses):
        return B.csa_lse_merge(outs, lses)


def torch_gather(group=None) -> Callable[[Tensor], List[Tensor]]:
    """all_gather over a torch.distributed group: every rank's tensor, in rank order."""
    import torch.distributed as dist

    def gather(t: Tensor) -> List[Tensor]:
        t = t.contiguous()
        out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(out, t, group=group)
        return out

    return gather


# --------------------------------------------------------------------------
# Phases (each rank runs them in order; the exchanges sit between them)
# --------------------------------------------------------------------------

def local_pairs(part: Part, iq: Tensor, w: Tensor, K: int, ops=CudaOps) -> Tuple[Tensor, Tensor]:
    """Step 1: the slice's top K as (score, global id) pairs, [B, 1, K] each."""
    scores = ops.index_score(part.cache, iq, w)
    idx = ops.topk(part.cache, scores, K)
    return ops.select_pairs(part.cache, scores, idx, part.row0)


def global_selection(all_scores: Sequence[Tensor], all_ids: Sequence[Tensor], K: int, ops=CudaOps) -> Tensor:
    """Step 3: the global top K of every rank's pairs -> [B, 1, K] global ids,
    ascending (the ranks' lists are in slice order), -1 padded."""
    ps = torch.cat([s.reshape(s.shape[0], -1) for s in all_scores], dim=-1)
    pi = torch.cat([i.reshape(i.shape[0], -1) for i in all_ids], dim=-1)
    return ops.topk_pairs(ps, pi, K).reshape(ps.shape[0], 1, K)


def local_attention(part: Part, q: Tensor, idx_global: Tensor, scale: float, ops=CudaOps) -> Tuple[Tensor, Tensor]:
    """Step 4: attention over the selected rows in this slice -> (out, lse)."""
    idx = ops.ids_window(idx_global, part.row0, part.row0 + part.rows)
    return ops.attend(part.cache, q, idx, scale)


def merge(all_out: Sequence[Tensor], all_lse: Sequence[Tensor], ops=CudaOps) -> Tuple[Tensor, Tensor]:
    """Step 5: the log-sum-exp merge of every rank's partial result."""
    return ops.lse_merge(torch.stack(list(all_out)), torch.stack(list(all_lse)))


# --------------------------------------------------------------------------
# A layer on one rank
# --------------------------------------------------------------------------

def layer_step(part: Part, q: Tensor, K: int, scale: float, gather: Callable[[Tensor], List[Tensor]],
               iq: Optional[Tensor] = None, w: Optional[Tensor] = None, idx_global: Optional[Tensor] = None,
               ops=CudaOps) -> Tuple[Tensor, Tensor, Tensor]:
    """One Full or Reindex layer (iq and w given: a fresh selection over every
    row of the sequence) or Reuse layer (idx_global given) on this rank.
    Returns (idx_global [B, 1, K], out [B, 1, H, D], lse [B, 1, H]), the same on
    every rank."""
    if idx_global is None:
        ps, pi = local_pairs(part, iq, w, K, ops)
        idx_global = global_selection(gather(ps), gather(pi), K, ops)
    out, lse = local_attention(part, q, idx_global, scale, ops)
    out, lse = merge(gather(out), gather(lse), ops)
    return idx_global, out, lse
