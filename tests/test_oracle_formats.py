"""Pins of the oracle's number formats and of the a1 quantiser (CPU only).

Each check compares the oracle with something other than itself: the pages'
printed facts (tests/golden), torch's own FP8/bf16 casts, exhaustive sweeps
against an independent threshold formulation, and closed-form invariants.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

FMT = {k: int(v) for k, v in read_golden("fp4_format.txt")}


def torch_e4m3_table():
    """E4M3 byte -> value via torch's float8_e4m3fn cast (NaN for 0x7F/0xFF)."""
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_decode_matches_printed_grid():
    for code, val in read_golden("e2m1_grid.txt"):
        got = oracle.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_decode_matches_torch_cast():
    t = torch_e4m3_table()
    for byte in range(256):
        got = oracle.e4m3_value(byte)
        if np.isnan(t[byte]):
            assert math.isnan(got)
        else:
            assert got == t[byte], byte
    assert oracle.e4m3_value(0x7E) == FMT["e4m3_max"]
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_bf16_decode_matches_torch_cast():
    bits = torch.arange(0, 65536, 97, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits.tolist(), ref):
        got = oracle.bf16_value(b)
        if np.isnan(r):
            assert math.isnan(got)
        else:
            assert got == r


def test_entry_size_matches_pages():
    D = FMT["entry_dim"]
    x = np.zeros((1, D), np.uint16)
    codes, scales = oracle.quantize_rows(x)
    assert codes.nbytes == FMT["entry_code_bytes"]
    assert scales.nbytes == FMT["entry_scale_bytes"]
    assert codes.nbytes + scales.nbytes == FMT["entry_bytes"]
    assert D // scales.shape[-1] == FMT["channels_per_scale"]
    # The pages' per-token accounting (3 Full layers at m=2 plus 1 at m=1).
    per_entry = FMT["entry_bytes"] + FMT["indexer_entry_bytes_mxfp4"]
    assert 3 * per_entry // 2 + per_entry == FMT["bytes_per_token"]
    assert FMT["pool_blocks"] * FMT["pool_block"] == FMT["pool_candidates"]


# ---------------------------------------------------------------------------
# Independent formulation of the rounding rules: sorted value table from torch
# plus midpoint thresholds (not the oracle's nearest-by-distance search).
# ---------------------------------------------------------------------------

def _e4m3_nonneg_sorted():
    t = torch_e4m3_table()
    codes = np.arange(0x7F)           # 0x00..0x7E: the finite non-negative values, ascending
    return codes, t[codes]


def ref_scale_byte(amax: float) -> int:
    """RNE(amax/6) onto E4M3, saturating at 448, via exact rational midpoints."""
    codes, vals = _e4m3_nonneg_sorted()
    target = Fraction(amax) / 6
    if target >= Fraction(float(vals[-1])):
        return int(codes[-1])
    hi = int(np.searchsorted(vals, float(target), side="left"))
    # refine with exact rationals around the float search position
    hi = max(1, min(hi, len(vals) - 1))
    while hi > 1 and Fraction(float(vals[hi - 1])) > target:
        hi -= 1
    while hi < len(vals) - 1 and Fraction(float(vals[hi])) < target:
        hi += 1
    lo = hi - 1
    vlo, vhi = Fraction(float(vals[lo])), Fraction(float(vals[hi]))
    if target <= vlo:
        return int(codes[lo])
    mid = (vlo + vhi) / 2
    if target < mid:
        return int(codes[lo])
    if target > mid:
        return int(codes[hi])
    return int(codes[lo]) if codes[lo] % 2 == 0 else int(codes[hi])


def ref_code_mag(ax: np.ndarray, s: float) -> np.ndarray:
    """E2M1 magnitude code of |x|/s by threshold counting with ties to even codes:
    cross the midpoint between codes k and k+1 only when strictly above it if k
    is even, or when at/above it if k is odd."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    code = np.zeros(ax.shape, np.int64)
    for k in range(7):
        mid = (grid[k] + grid[k + 1]) / 2 * s      # exact in float64
        code += (ax > mid) if k % 2 == 0 else (ax >= mid)
    return code


def all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals)
    return bits[ok], vals[ok]


@pytest.mark.parametrize("sbyte", [0x01, 0x07, 0x08, 0x20, 0x38, 0x3B, 0x55, 0x7E])
def test_code_rounding_exhaustive_over_bf16(sbyte):
    """Every finite bf16 value against a fixed E4M3 scale: oracle == thresholds."""
    s = oracle.e4m3_value(sbyte)
    bits, vals = all_finite_bf16()
    ref = ref_code_mag(np.abs(vals), s)
    L = oracle.lib()
    got = np.array([L.oracle_e2m1_round_ratio(abs(v), s) for v in vals], np.int64)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(bits[i]), vals[i], got[i], ref[i]) for i in bad[:5]]


def test_scale_rounding_exhaustive_over_bf16_amax():
    bits, vals = all_finite_bf16()
    L = oracle.lib()
    pos = vals[vals >= 0]
    # every 3rd positive finite bf16 magnitude (about 11k values), plus the
    # neighbourhood of the saturation point
    sample = np.concatenate([pos[::3], pos[(pos > 2500) & (pos < 3000)]])
    for a in sample:
        assert L.oracle_e4m3_round_ratio(float(a), 6.0) == ref_scale_byte(float(a)), a


def test_quantize_group_invariants():
    """Grid membership, half-spacing error bound, sign symmetry and power-of-two
    equivariance of whole groups drawn at many magnitudes."""
    from fp4_compressed_sparse_append_b300 import workloads as W
    grid = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    spacing_above = {0.0: 0.5, 0.5: 0.5, 1.0: 0.5, 1.5: 0.5, 2.0: 1.0, 3.0: 1.0, 4.0: 2.0, 6.0: 2.0}
    for tag, std in enumerate([1e-4, 0.01, 1.0, 7.5, 100.0, 300.0]):
        x = W.random_bf16_bits((64, 64), seed=1, tag=tag, std=std).numpy().view(np.uint16)
        codes, scales = oracle.quantize_rows(x)
        dq = oracle.dequantize_rows(codes, scales)
        xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        for r in range(x.shape[0]):
            for g in range(x.shape[1] // 16):
                s = oracle.e4m3_value(int(scales[r, g]))
                amax = np.abs(xv[r, g * 16:(g + 1) * 16]).max()
                assert scales[r, g] == ref_scale_byte(amax)
                if s == 0:
                    assert np.all(dq[r, g * 16:(g + 1) * 16] == 0)
                    continue
                for i in range(16):
                    m = abs(dq[r, g * 16 + i]) / s
                    assert m in grid
                    err = abs(abs(xv[r, g * 16 + i]) - abs(dq[r, g * 16 + i]))
                    if abs(xv[r, g * 16 + i]) <= 6 * s:
                        assert err <= spacing_above[m] / 2 * s
        # sign symmetry: flipping every sign flips exactly the code sign bits
        c2, s2 = oracle.quantize_rows(x ^ np.uint16(0x8000))
        assert np.array_equal(s2, scales)
        live = np.repeat(scales != 0, 8, axis=1)          # code bytes of groups with a scale
        assert np.array_equal(c2[live], codes[live] ^ np.uint8(0x88))
        assert not c2[~live].any() and not codes[~live].any()
        # multiplying by 4 (two exponent steps, no saturation at these sizes)
        if std <= 100.0:
            x4 = x.astype(np.int32) + ((x & 0x7F80) != 0) * (2 << 7)
            x4 = x4.astype(np.uint16)
            c4, s4 = oracle.quantize_rows(x4)
            dq4 = oracle.dequantize_rows(c4, s4)
            normal_groups = ((x.reshape(64, -1, 16) & 0x7F80) != 0).all(axis=2)
            for r, g in zip(*np.nonzero(normal_groups)):
                if 0x09 <= scales[r, g] <= 0x6E:   # normal scale both before and after x4
                    assert np.array_equal(dq4[r, g * 16:(g + 1) * 16], 4 * dq[r, g * 16:(g + 1) * 16])


def test_saturation_at_2688():
    """The pages give FP4-with-scale's range as 2,688 = 6 x 448."""
    D = 16
    top = FMT["fp4_with_scale_max"]
    for amax, expect in [(2688.0, 2688.0), (3000.0, 2688.0), (1.0e6, 2688.0)]:
        x = torch.zeros(1, D, dtype=torch.float32)
        x[0, 3] = amax
        x[0, 4] = -amax
        bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        codes, scales = oracle.quantize_rows(bits)
        dq = oracle.dequantize_rows(codes, scales)
        assert scales[0, 0] == 0x7E
        assert dq[0, 3] == expect == top
        assert dq[0, 4] == -expect


def test_negative_zero_and_zero_group():
    x = np.zeros((1, 32), np.uint16)
    x[0, 0] = 0x8000                       # -0 in a group with a nonzero scale
    x[0, 1] = 0x3F80                       # 1.0
    x[0, 2] = 0xB400                       # -2^-23 (rounds to magnitude 0, sign kept)
    codes, scales = oracle.quantize_rows(x)
    assert scales[0, 0] == 0x23            # RNE(1/6) = 0.171875 = 1.375 * 2^-3
    assert codes[0, 0] & 0xF == 0x8
    assert codes[0, 1] & 0xF == 0x8        # channel 2 (low nibble of byte 1)
    # second group is all zero -> scale 0 and all-zero codes
    assert scales[0, 1] == 0
    assert np.all(codes[0, 8:] == 0)
