"""Pins of the oracle's MXFP4 indexer keys (CPU only).

"G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache entries, and why
they're safe": an indexer K entry is 128 values x 4 bits plus one 8-bit scale
per 32 values (68 B), the OCP MXFP4 format.  The oracle's rule: X = floor(log2
amax) - 2 clamped to [-8, 6], scale byte X + 127, codes nearest E2M1 to
|x| / 2^X with ties to the even code and 6 beyond.  Each check compares the
oracle with something other than itself: exact rational brute force over the
printed E2M1 grid (tests/golden), torch's E4M3 cast, the already-pinned E4M3
scoring path, and a float64 numpy product.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

GRID = {int(c): float(v) for c, v in read_golden("e2m1_grid.txt")}
MAGS = [Fraction(GRID[c]) for c in range(8)]


def ref_exponent(amax: Fraction) -> int:
    """Largest t with 2^(t+2) <= amax, clamped to [-8, 6]; -8 for 0 (exact arithmetic)."""
    if amax == 0:
        return -8
    t = -200
    while Fraction(2) ** (t + 3) <= amax:
        t += 1
    return max(-8, min(6, t))


def ref_code(x: Fraction, X: int, negative: bool) -> int:
    """Nearest grid magnitude to |x| / 2^X, ties to the even code, 6 beyond; sign bit kept."""
    q = abs(x) / Fraction(2) ** X
    best, best_d = 0, None
    for c, m in enumerate(MAGS):
        d = abs(q - m)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0 and best % 2 == 1):
            best, best_d = c, d
    if q >= 6:
        best = 7
    return best | (8 if negative else 0)


def ref_quantize_block(vals):
    fr = [Fraction(v) for v in vals]
    X = ref_exponent(max(abs(v) for v in fr))
    codes = [ref_code(v, X, np.signbit(vals[i])) for i, v in enumerate(fr)]
    return X, codes


def unpack(codes_row):
    out = []
    for byte in codes_row:
        out += [int(byte) & 0xF, int(byte) >> 4]
    return out


def test_block_exponent_matches_exact_rule():
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(2000) * np.exp2(rng.integers(-20, 20, 2000)))
    for k in range(-14, 14):                         # powers of two and their neighbours
        p = 2.0 ** k
        vals += [p, np.nextafter(p, 0.0), np.nextafter(p, np.inf)]
    vals += [0.0, 1e30, 1e-30]
    for v in vals:
        a = abs(float(v))
        assert oracle.mx_exponent(a) == ref_exponent(Fraction(a)), a


@pytest.mark.parametrize("scale_pow", [-12, -5, 0, 3, 9])
def test_quantize_matches_brute_force(scale_pow):
    rng = np.random.default_rng(100 + scale_pow)
    x = (rng.standard_normal((6, 128)) * 2.0 ** scale_pow)
    x[0, :32] = 0.0                                   # an all-zero block
    x[1, 5] = -0.0
    x[2, :32] = 2.0 ** scale_pow * np.array(MAGS + MAGS[::-1] + MAGS + MAGS[::-1], float)  # grid points
    x = x.astype(np.float32).astype(np.float64)       # float32-representable reals
    codes, scales = oracle.mx_quantize(x)
    for r in range(x.shape[0]):
        got = unpack(codes[r])
        for blk in range(4):
            X, want = ref_quantize_block(x[r, blk * 32:(blk + 1) * 32])
            assert scales[r, blk] == X + 127, (r, blk)
            assert got[blk * 32:(blk + 1) * 32] == want, (r, blk)


def test_decoded_keys_are_exact_e4m3_values():
    # every code under every in-range scale decodes to an exact E4M3 value
    codes = np.arange(256, dtype=np.uint8).reshape(1, 256)[:, :64].repeat(15, axis=0)   # 128 nibbles per row
    scales = (np.arange(-8, 7) + 127).astype(np.uint8)[:, None].repeat(4, axis=1)
    v = oracle.mx_dequantize(codes, scales)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.abs(t), np.abs(v))
    for X in range(-8, 7):
        row = X + 8
        assert np.isclose(np.abs(v[row]).max(), 6.0 * 2.0 ** X)


def test_mx_scores_equal_e4m3_scores_of_the_decoded_keys():
    rng = np.random.default_rng(7)
    n, HI, DI = 300, 8, 128
    x = rng.standard_normal((n, DI)) * np.exp2(rng.integers(-3, 3, (n, 1)))
    codes, scales = oracle.mx_quantize(x)
    keys = oracle.mx_pack(codes, scales)
    dec = oracle.mx_dequantize(codes, scales)
    e4 = torch.from_numpy(dec.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    iq = torch.from_numpy(rng.standard_normal((HI, DI)).astype(np.float32)).to(torch.float8_e4m3fn)
    iq = iq.view(torch.uint8).numpy()
    w = rng.random(HI).astype(np.float32)
    rows = np.arange(n)
    assert np.array_equal(oracle.index_scores_mx(iq, w, keys, rows), oracle.index_scores(iq, w, e4, rows))


def test_projection_to_mx_matches_float64_product():
    rng = np.random.default_rng(9)
    D, DI = 256, 128
    xb = torch.from_numpy(rng.standard_normal((5, D)).astype(np.float32)).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows(xb.view(torch.int16).numpy())
    wf = torch.from_numpy((rng.standard_normal((D, DI)) / np.sqrt(D)).astype(np.float32)).to(torch.bfloat16)
    keys = oracle.project_ikeys_mx(codes, scales, wf.view(torch.int16).numpy())
    exact = oracle.dequantize_rows(codes, scales) @ wf.to(torch.float64).numpy()   # exact for these sizes
    kc, ks = oracle.mx_unpack(keys, DI)
    for r in range(5):
        got = unpack(kc[r])
        for blk in range(DI // 32):
            X, want = ref_quantize_block(exact[r, blk * 32:(blk + 1) * 32])
            assert ks[r, blk] == X + 127
            assert got[blk * 32:(blk + 1) * 32] == want
