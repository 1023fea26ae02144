"""Seeded synthetic inputs for the CSA2 decode step.

This module only draws random numbers and lays them out in the shapes the
step consumes. It holds none of the method's arithmetic: no quantiser, no
score, no selection and no attention. Both the CUDA path (through the
binding) and the CPU oracle (through the tests) take their inputs from here.

Randomness comes from ``torch.Generator`` streams, one per tensor, seeded by a
splitmix64 mix of (seed, tensor tag, sequence index).  Draws made on a CUDA
device differ from draws made on the CPU; a test that compares the two paths
draws once and copies the same bytes to both sides.

Conversion of the normal draws to bf16 and to FP8 E4M3 bytes uses torch's own
dtype casts (round to nearest even); those bytes are *inputs* to the step.

Workloads (the shapes of long-context agent decoding: a 1M-token window, one
shared 512-dim latent per cached position, 64 query heads and a 64x128 FP8
indexer):

=================  ==  ========  ==  ===  ==  ===  ====  =  =========================
name               B   context   H   D    HI  DI   K     P  layers
=================  ==  ========  ==  ===  ==  ===  ====  =  =========================
tiny_full          1   4096      16  128  4   64   256   1  Full
full_64k           8   65536     64  512  64  128  2048  1  Full (1% outlier channels)
chain_128k         32  131072    64  512  64  128  2048  1  Full, 3x Reindex, 4x Reuse
hier_1m            1   1048576   64  512  64  128  2048  1  Full+pool, 7x Reindex(pool)
verify_append_32k  64  32768     64  512  64  128  2048  6  append 6 rows, then Full
full_64k_swa       8   65536     64  512  64  128  2048  1  Full + 128-row local window
full_64k_mx        8   65536     64  512  64  128  2048  1  Full, MXFP4 indexer keys (68 B)
chain_128k_mx      32  131072    64  512  64  128  2048  1  as chain_128k, MXFP4 indexer keys
verify_project_32k 64  32768     64  512  64  128  2048  6  as verify_append_32k, keys projected
=================  ==  ========  ==  ===  ==  ===  ====  =  =========================
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch

FULL, REINDEX, REUSE = 0, 1, 2
MODE_NAMES = {FULL: "full", REINDEX: "reindex", REUSE: "reuse"}

POOL_BLOCK = 8          # positions per pool block (hierarchical indexer)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                  # sequences in the batch
    L: int                  # cached rows per sequence before the step
    H: int                  # main query heads
    D: int                  # latent dim (FP4 row = D/2 code bytes + D/16 scale bytes)
    HI: int                 # indexer heads
    DI: int                 # indexer key dim (FP8 E4M3 bytes per key)
    K: int                  # top-K
    P: int = 1              # query positions per sequence (causal)
    layers: Tuple[int, ...] = (FULL,)
    pool_blocks: int = 0    # >0: the first Full layer also keeps this many 8-row blocks,
                            # and Reindex layers rescore only that pool
    outlier_channels: int = 0   # latent channels scaled x8 (same channels in every row)
    planted: int = 0        # length of a planted high-similarity block (0 = none)
    n_append: int = 0       # rows appended (quantised) at the start of the step
    window: int = 0         # >0: every query also attends to this many local FP8 rows
    project: bool = False   # indexer keys projected from the stored rows by a seeded [D][DI] matrix
    key_format: str = "e4m3"  # "mxfp4": E2M1 codes + one UE8M0 scale per 32 key channels (d_index 128)

    @property
    def capacity(self) -> int:
        return self.L + self.n_append

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def length_after_append(self) -> int:
        return self.L + self.n_append

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny_full": Workload("tiny_full", B=1, L=4096, H=16, D=128, HI=4, DI=64, K=256),
    "full_64k": Workload("full_64k", B=8, L=65536, H=64, D=512, HI=64, DI=128, K=2048,
                         outlier_channels=5),
    "chain_128k": Workload("chain_128k", B=32, L=131072, H=64, D=512, HI=64, DI=128, K=2048,
                           layers=(FULL, REINDEX, REINDEX, REINDEX, REUSE, REUSE, REUSE, REUSE)),
    "hier_1m": Workload("hier_1m", B=1, L=1048576, H=64, D=512, HI=64, DI=128, K=2048,
                        layers=(FULL,) + (REINDEX,) * 7, pool_blocks=2048, planted=512),
    "verify_append_32k": Workload("verify_append_32k", B=64, L=32768, H=64, D=512, HI=64,
                                  DI=128, K=2048, P=6, n_append=6),
    "full_64k_swa": Workload("full_64k_swa", B=8, L=65536, H=64, D=512, HI=64, DI=128, K=2048,
                             outlier_channels=5, window=128),
    "verify_project_32k": Workload("verify_project_32k", B=64, L=32768, H=64, D=512, HI=64,
                                   DI=128, K=2048, P=6, n_append=6, project=True),
    "full_64k_mx": Workload("full_64k_mx", B=8, L=65536, H=64, D=512, HI=64, DI=128, K=2048,
                            outlier_channels=5, key_format="mxfp4"),
    "chain_128k_mx": Workload("chain_128k_mx", B=32, L=131072, H=64, D=512, HI=64, DI=128, K=2048,
                              layers=(FULL, REINDEX, REINDEX, REINDEX, REUSE, REUSE, REUSE, REUSE),
                              key_format="mxfp4"),
}

# Tensor tags for the per-tensor streams.
_T_LATENT, _T_IKEY, _T_Q, _T_IQ, _T_W, _T_NEWROW, _T_NEWIKEY, _T_OUTLIER, _T_PLANT, _T_LOCAL, _T_WIK, _T_MXKEY = range(12)


def _mix(*vals: int) -> int:
    """splitmix64 over a tuple of integers -> a 63-bit torch seed."""
    x = 0x9E3779B97F4A7C15
    for v in vals:
        x = (x ^ (v & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


def _gen(device, *tag: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*tag))
    return g


def _randn(shape, device, *tag) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(device, *tag), device=device, dtype=torch.float32)


def to_bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 (torch RNE cast), returned as the raw bits in an int16 tensor."""
    return x.to(torch.bfloat16).view(torch.int16)


def to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> FP8 E4M3 (torch RNE cast), returned as raw bytes (uint8)."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def outlier_channels(wl: Workload, seed: int) -> torch.Tensor:
    """The latent channels that carry x8 outliers (CPU int64 tensor)."""
    if wl.outlier_channels == 0:
        return torch.zeros(0, dtype=torch.int64)
    g = _gen("cpu", seed, _T_OUTLIER)
    return torch.randperm(wl.D, generator=g)[: wl.outlier_channels].sort().values


def planted_offset(wl: Workload, seed: int) -> int:
    """Start row of the planted block (unaligned), or -1 if the workload has none."""
    if wl.planted == 0:
        return -1
    g = _gen("cpu", seed, _T_PLANT, 0)
    return int(torch.randint(0, wl.L - wl.planted + 1, (1,), generator=g).item())


def _planted_centres(wl: Workload, seed: int, device) -> Tuple[torch.Tensor, torch.Tensor]:
    c_ik = _randn((wl.DI,), device, seed, _T_PLANT, 1)
    c_lat = _randn((wl.D,), device, seed, _T_PLANT, 2)
    return c_ik, c_lat


def cache_rows(wl: Workload, seed: int, b: int, device="cpu",
               rows: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Latents (bf16 bits, [n, D]) and indexer keys (E4M3 bytes, [n, DI]) of sequence b.

    ``rows=(r0, r1)`` restricts the draw to rows [r0, r1) of the sequence; rows
    are drawn in fixed chunks of 65536, so any sub-range reproduces the same
    values as the full draw on the same device.
    """
    r0, r1 = rows if rows is not None else (0, wl.L)
    CH = 65536
    lat_parts, ik_parts = [], []
    out_ch = outlier_channels(wl, seed).to(device)
    off = planted_offset(wl, seed)
    if off >= 0:
        c_ik, c_lat = _planted_centres(wl, seed, device)
    for c0 in range((r0 // CH) * CH, r1, CH):
        c1 = min(c0 + CH, wl.L)
        lat = _randn((c1 - c0, wl.D), device, seed, _T_LATENT, b, c0)
        ik = _randn((c1 - c0, wl.DI), device, seed, _T_IKEY, b, c0)
        if out_ch.numel():
            lat[:, out_ch] *= 8.0
        if off >= 0:
            p0, p1 = max(off, c0), min(off + wl.planted, c1)
            if p0 < p1:
                z_lat = lat[p0 - c0:p1 - c0].clone()
                z_ik = ik[p0 - c0:p1 - c0].clone()
                lat[p0 - c0:p1 - c0] = c_lat + 0.25 * z_lat
                ik[p0 - c0:p1 - c0] = c_ik + 0.25 * z_ik
        s0, s1 = max(r0, c0) - c0, min(r1, c1) - c0
        lat_parts.append(to_bf16_bits(lat[s0:s1]))
        if wl.key_format == "mxfp4":
            ik_parts.append(random_mx_keys(c1 - c0, wl.DI, device, seed, b, c0)[s0:s1])
        else:
            ik_parts.append(to_e4m3_bytes(ik[s0:s1]))
    return torch.cat(lat_parts), torch.cat(ik_parts)


def layer_inputs(wl: Workload, seed: int, layer: int, device="cpu") -> Dict[str, torch.Tensor]:
    """Per-layer query inputs for all B sequences and P positions.

    q  : bf16 bits  [B, P, H, D]   main query, N(0,1)
    iq : E4M3 bytes [B, P, HI, DI] indexer query, N(0,1)
    w  : fp32       [B, P, HI]     per-head indexer weights, U(0,1)
    """
    B, P = wl.B, wl.P
    q = _randn((B, P, wl.H, wl.D), device, seed, _T_Q, layer)
    iq = _randn((B, P, wl.HI, wl.DI), device, seed, _T_IQ, layer)
    w = torch.rand((B, P, wl.HI), generator=_gen(device, seed, _T_W, layer), device=device)
    if wl.planted:
        # Planted block: its keys sit near c_ik, and every layer's indexer heads
        # lean towards c_ik, so the block is relevant to every layer's query.
        c_ik, c_lat = _planted_centres(wl, seed, device)
        iq = (iq + c_ik) / math.sqrt(2.0)
        q = q + c_lat / math.sqrt(2.0)
    return {"q": to_bf16_bits(q), "iq": to_e4m3_bytes(iq), "w": w}


def append_rows(wl: Workload, seed: int, device="cpu") -> Dict[str, torch.Tensor]:
    """Rows appended at the start of the step: bf16 latents [B, n, D], ikeys [B, n, key bytes]."""
    n = wl.n_append
    lat = _randn((wl.B, n, wl.D), device, seed, _T_NEWROW)
    ik = _randn((wl.B, n, wl.DI), device, seed, _T_NEWIKEY)
    out_ch = outlier_channels(wl, seed).to(device)
    if out_ch.numel():
        lat[..., out_ch] *= 8.0
    if wl.key_format == "mxfp4":
        keys = random_mx_keys(wl.B * n, wl.DI, device, seed, _T_NEWIKEY).view(wl.B, n, -1)
    else:
        keys = to_e4m3_bytes(ik)
    return {"rows": to_bf16_bits(lat), "ikeys": keys}


def key_bytes(wl: Workload) -> int:
    """Bytes of one indexer key row as the tests and the C ABI's append take it."""
    return wl.DI // 2 + wl.DI // 32 if wl.key_format == "mxfp4" else wl.DI


def random_mx_keys(n: int, DI: int, device, *tag) -> torch.Tensor:
    """Packed MXFP4 key rows [n, DI/2 + DI/32]: uniform code bytes (every E2M1
    code), then scale bytes uniform over [119, 133] (block exponents -8..6)."""
    g = _gen(device, _T_MXKEY, *tag)
    codes = torch.randint(0, 256, (n, DI // 2), generator=g, device=device, dtype=torch.int32)
    scales = torch.randint(119, 134, (n, DI // 32), generator=g, device=device, dtype=torch.int32)
    return torch.cat([codes, scales], dim=1).to(torch.uint8)


def ikey_projection(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    """The [D][DI] matrix that projects stored rows to indexer keys: N(0, 1/D)
    in bf16 (bits as int16), so a key channel has about the spread of a latent."""
    return to_bf16_bits(_randn((wl.D, wl.DI), device, seed, _T_WIK) / math.sqrt(wl.D))


def local_rows(wl: Workload, seed: int, device="cpu", n: Optional[int] = None) -> torch.Tensor:
    """The local window's rows of every sequence: E4M3 bytes [B, n, D] (default
    n = window + P - 1, enough for the full window of each of the P positions),
    latents drawn like the cached rows (N(0,1), the same outlier channels x8)."""
    n = wl.window + wl.P - 1 if n is None else n
    lat = _randn((wl.B, n, wl.D), device, seed, _T_LOCAL)
    out_ch = outlier_channels(wl, seed).to(device)
    if out_ch.numel():
        lat[..., out_ch] *= 8.0
    return to_e4m3_bytes(lat)


def random_bf16_bits(shape, seed: int, tag: int = 0, device="cpu", std: float = 1.0) -> torch.Tensor:
    """Generic N(0, std^2) bf16 bits for edge-case tests."""
    return to_bf16_bits(_randn(shape, device, seed, 0x5EED, tag) * std)


def random_e4m3_bytes(shape, seed: int, tag: int = 0, device="cpu", std: float = 1.0) -> torch.Tensor:
    return to_e4m3_bytes(_randn(shape, device, seed, 0x5EEE, tag) * std)


def random_uniform(shape, seed: int, tag: int = 0, device="cpu") -> torch.Tensor:
    return torch.rand(shape, generator=_gen(device, seed, 0x5EEF, tag), device=device)


def random_scores(shape, seed: int, tag: int = 0, device="cpu") -> torch.Tensor:
    """fp32 scores for selection tests: N(0,1) draws."""
    return _randn(shape, device, seed, 0x5EF0, tag)


def random_ints(shape, low: int, high: int, seed: int, tag: int = 0, device="cpu") -> torch.Tensor:
    return torch.randint(low, high, shape, generator=_gen(device, seed, 0x5EF1, tag),
                         device=device, dtype=torch.int64)
