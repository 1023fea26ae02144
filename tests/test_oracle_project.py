"""Pins of the oracle's projected indexer keys (CPU only).

"G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
index, select": the indexer's keys are a projection of the main cache entries.
The oracle computes ik[j] = E4M3(sum_c v[c] * w[c][j]) from the stored FP4 row.
Each check compares it with something other than itself: torch's own
float8_e4m3fn cast, the printed E2M1 grid (tests/golden), a float64 numpy
product, and closed-form properties (identity and one-entry projections,
linearity, sign symmetry, saturation).
"""
import numpy as np
import torch

import oracle
from conftest import read_golden

GRID = {int(c): float(v) for c, v in read_golden("e2m1_grid.txt")}


def torch_e4m3(x: np.ndarray) -> np.ndarray:
    """E4M3 bytes of float32-representable values by torch's cast (RNE)."""
    t = torch.from_numpy(np.asarray(x, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def as_sum(b: np.ndarray) -> np.ndarray:
    """A sum of products is +0 when it is zero (the sign of -0 inputs is lost)."""
    b = np.array(b, np.uint8)
    b[b == 0x80] = 0
    return b


def e4m3_values(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_by_grid(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Rows decoded with the printed grid and torch's E4M3 decode (not the oracle's)."""
    n, half = codes.shape
    D = half * 2
    lo, hi = codes & 0xF, codes >> 4
    nib = np.empty((n, D), np.int64)
    nib[:, 0::2], nib[:, 1::2] = lo, hi
    vals = np.vectorize(GRID.get)(nib).astype(np.float64)
    sc = e4m3_values(scales)
    return vals * np.repeat(sc, 16, axis=1)


def rows(n, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((n, D), generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy()
    return oracle.quantize_rows(x)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_signed_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(3)
    # random float32 values across the E4M3 range, both signs
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 8, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    got = np.array([oracle.e4m3_round(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, torch_e4m3(x))
    # exact midpoints between neighbouring values: ties go to the even code
    pos = np.sort(e4m3_values(np.arange(0x7F, dtype=np.uint8)))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)
    for m in np.concatenate([mids, -mids]):
        assert oracle.e4m3_round(float(m)) == int(torch_e4m3(np.array([m]))[0])


def test_saturation_and_signed_zero():
    assert oracle.e4m3_round(448.0) == 0x7E
    assert oracle.e4m3_round(464.0) == 0x7E          # the midpoint towards 480, which E4M3 lacks
    assert oracle.e4m3_round(1.0e6) == 0x7E
    assert oracle.e4m3_round(-1.0e6) == 0xFE
    assert oracle.e4m3_round(0.0) == 0x00
    assert oracle.e4m3_round(-1.0e-9) == 0x80         # rounds to zero, keeps the sign


def test_identity_projection_rounds_each_channel():
    D, DI = 128, 64
    codes, scales = rows(5, D, seed=1)
    w = np.zeros((D, DI), np.float32)
    w[np.arange(DI), np.arange(DI)] = 1.0
    ik = oracle.project_ikeys(codes, scales, bf16_bits(w))
    v = dequant_by_grid(codes, scales)[:, :DI]
    assert np.abs(v).max() <= 448.0
    assert np.array_equal(ik, as_sum(torch_e4m3(v)))


def test_one_entry_per_output_column():
    D, DI = 256, 128
    codes, scales = rows(4, D, seed=2, std=3.0)
    rng = np.random.default_rng(4)
    src = rng.permutation(D)[:DI]
    wv = bf16_bits(rng.standard_normal(DI).astype(np.float32) * 4.0)
    w = np.zeros((D, DI), np.uint16)
    w[src, np.arange(DI)] = wv
    ik = oracle.project_ikeys(codes, scales, w)
    v = dequant_by_grid(codes, scales)
    wf = torch.from_numpy(wv.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    prod = v[:, src] * wf[None, :]                    # exact in float32 (8 + 6 significant bits)
    prod = np.clip(prod, -448.0, 448.0)
    assert np.array_equal(ik, as_sum(torch_e4m3(prod)))


def test_random_projection_matches_float64_product():
    D, DI = 512, 128
    codes, scales = rows(6, D, seed=5)
    rng = np.random.default_rng(6)
    w = bf16_bits(rng.standard_normal((D, DI)).astype(np.float32) / np.sqrt(D))
    ik = oracle.project_ikeys(codes, scales, w)
    wf = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    exact = dequant_by_grid(codes, scales) @ wf        # float64; exact for these magnitudes
    ref = as_sum(torch_e4m3(exact.astype(np.float32)))  # float64 -> float32 -> E4M3
    diff = ik != ref
    # a mismatch can only come from the float32 step landing on a rounding
    # midpoint: then the float64 value must sit within a float32 ulp of one
    for r, j in zip(*np.nonzero(diff)):
        x = abs(exact[r, j])
        lo, hi = sorted(e4m3_values(np.array([ik[r, j] & 0x7F, ref[r, j] & 0x7F], np.uint8)))
        assert abs(x - (lo + hi) / 2) <= 2.0 ** -23 * x, (r, j, x)
    assert diff.sum() <= 2


def test_linearity_and_sign():
    D, DI = 128, 32
    codes, scales = rows(3, D, seed=7)
    rng = np.random.default_rng(8)
    wf = rng.standard_normal((D, DI)).astype(np.float32) / np.sqrt(D)
    ik1 = oracle.project_ikeys(codes, scales, bf16_bits(wf))
    ik2 = oracle.project_ikeys(codes, scales, bf16_bits(2.0 * wf))   # exact doubling in bf16
    ikn = oracle.project_ikeys(codes, scales, bf16_bits(-wf))
    v1, v2 = e4m3_values(ik1), e4m3_values(ik2)
    normal = (np.abs(v1) >= 2.0 ** -6) & (np.abs(v1) <= 224.0)
    assert normal.sum() > 0.8 * v1.size
    assert np.array_equal(v2[normal], 2.0 * v1[normal])
    nz = (ik1 & 0x7F) != 0
    assert np.array_equal(ikn[nz], ik1[nz] ^ 0x80)
