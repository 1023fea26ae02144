"""Pins of the oracle's persistent cache records (CPU only).

"G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache entries, and why
they're safe", the derivation of the 890 bytes per token: an entry is its main
entry (288 B) and its MXFP4 indexer entry (68 B); a cache layer with
compression m keeps one entry per m tokens.  The checks compare the oracle with
the printed figures (tests/golden/persistent_cache.txt), with the meaning of a
record's fields (each decodes or scores like the stored row it came from, by
the printed E2M1 grid and torch's E4M3 decode, or the pinned scoring
functions), and with round trips.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

FIG = {k: int(v) for k, v in read_golden("persistent_cache.txt")}
GRID = {int(c): float(v) for c, v in read_golden("e2m1_grid.txt")}


def decode_main(codes, scales):
    """Main entries decoded by the printed grid and torch's E4M3 decode (not the oracle's)."""
    n, half = codes.shape
    nib = np.empty((n, half * 2), np.int64)
    nib[:, 0::2], nib[:, 1::2] = codes & 0xF, codes >> 4
    vals = np.vectorize(GRID.get)(nib).astype(np.float64)
    sc = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(sc, 16, axis=1)


def filled_cache(B, cap, D, DI, key_format, lengths, seed):
    g = torch.Generator().manual_seed(seed)
    c = oracle.Cache(B, cap, D, DI, key_format)
    n = max(lengths)
    rows = (torch.randn((B, n, D), generator=g) * 2).to(torch.bfloat16).view(torch.int16).numpy()
    if key_format == "mxfp4":
        kc, ks = oracle.mx_quantize(torch.randn((B * n, DI), generator=g).numpy().astype(np.float64))
        keys = oracle.mx_pack(kc, ks).reshape(B, n, -1)
    else:
        keys = torch.randn((B, n, DI), generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    c.append(rows, keys)
    c.lengths[:] = lengths          # ragged: rows past a length are not valid
    return c


def test_entry_bytes_match_the_printed_figures():
    D, DI = FIG["entry_dim"], FIG["index_dim"]
    assert oracle.record_bytes(D, DI, "mxfp4") == FIG["entry_bytes"]
    assert FIG["main_entry_bytes"] + FIG["indexer_entry_bytes"] == FIG["entry_bytes"]
    # the main part alone (an indexer key of 0 bytes is not a format; the E4M3
    # key of the same width adds DI bytes instead of DI/2 + DI/32)
    assert oracle.record_bytes(D, DI, "e4m3") - DI == FIG["main_entry_bytes"]


def test_bytes_per_token_match_the_printed_figures():
    e = FIG["entry_bytes"]
    enc = oracle.bytes_per_token([e] * FIG["encoder_full_layers"], [FIG["encoder_m"]] * FIG["encoder_full_layers"])
    dec = oracle.bytes_per_token([e] * FIG["decoder_full_layers"], [FIG["decoder_m"]] * FIG["decoder_full_layers"])
    assert enc == FIG["encoder_bytes_per_token"] and dec == FIG["decoder_bytes_per_token"]
    allb = oracle.bytes_per_token([e] * 4, [2, 2, 2, 1])
    assert allb == FIG["bytes_per_token"]
    # with E4M3 keys of the same width the entry grows by 128 - 68 bytes
    e8 = oracle.record_bytes(512, 128, "e4m3")
    assert oracle.bytes_per_token([e8] * 4, [2, 2, 2, 1]) == FIG["bytes_per_token"] + (128 - 68) * 2.5


@pytest.mark.parametrize("key_format,D,DI", [("mxfp4", 512, 128), ("e4m3", 256, 64), ("e4m3", 128, 32)])
def test_record_fields_decode_like_the_stored_rows(key_format, D, DI):
    B, cap = 3, 40
    lengths = [37, 20, 40]
    c = filled_cache(B, cap, D, DI, key_format, lengths, seed=11)
    rec = oracle.cache_spill(c, 0, cap)
    cb, sb = D // 2, D // 16
    assert rec.shape == (B, cap, oracle.record_bytes(D, DI, key_format))
    rng = np.random.default_rng(5)
    HI = 4
    iq = torch.from_numpy(rng.standard_normal((HI, DI)).astype(np.float32)).to(torch.float8_e4m3fn)
    iq = iq.view(torch.uint8).numpy()
    w = rng.random(HI).astype(np.float32)
    score = oracle.index_scores_mx if key_format == "mxfp4" else oracle.index_scores
    for b in range(B):
        L = lengths[b]
        got = decode_main(rec[b, :L, :cb], rec[b, :L, cb:cb + sb])
        want = decode_main(c.codes[b, :L], c.scales[b, :L])
        assert np.array_equal(got, want)
        rows = np.arange(L)
        assert np.array_equal(score(iq, w, rec[b, :L, cb + sb:], rows), score(iq, w, c.ikeys[b, :L], rows))
        assert not rec[b, L:].any()                                    # rows past the length are zeros


@pytest.mark.parametrize("key_format", ["mxfp4", "e4m3"])
def test_round_trip_and_windows(key_format):
    D, DI, B, cap = 256, 128 if key_format == "mxfp4" else 64, 2, 64
    lengths = [50, 33]
    c = filled_cache(B, cap, D, DI, key_format, lengths, seed=12)
    # the whole valid prefix, reloaded into an empty cache, is the same cache
    n = min(lengths)
    r = oracle.cache_spill(c, 0, n)
    e = oracle.Cache(B, cap, D, DI, key_format)
    assert oracle.cache_reload(e, r) == 0
    assert list(e.lengths) == [n, n]
    for t in ("codes", "scales", "ikeys"):
        assert np.array_equal(getattr(e, t)[:, :n], getattr(c, t)[:, :n])
    # windows concatenate: spill(0, k) ++ spill(k, n - k) == spill(0, n)
    k = 13
    assert np.array_equal(np.concatenate([oracle.cache_spill(c, 0, k), oracle.cache_spill(c, k, n - k)], 1), r)
    # reloading in two parts appends after the first
    e2 = oracle.Cache(B, cap, D, DI, key_format)
    oracle.cache_reload(e2, r[:, :k])
    oracle.cache_reload(e2, r[:, k:])
    for t in ("codes", "scales", "ikeys"):
        assert np.array_equal(getattr(e2, t), getattr(e, t))


def test_reload_leaves_a_full_sequence_unchanged():
    D, DI, B, cap = 128, 32, 2, 10
    c = filled_cache(B, cap, D, DI, "e4m3", [6, 6], seed=13)
    c.lengths[1] = 8
    before = [a.copy() for a in (c.codes, c.scales, c.ikeys)]
    rec = np.full((B, 3, oracle.record_bytes(D, DI)), 0x5A, np.uint8)
    assert oracle.cache_reload(c, rec) == 1                             # 8 + 3 > 10
    assert list(c.lengths) == [9, 8]
    assert np.array_equal(c.codes[1], before[0][1]) and np.array_equal(c.ikeys[1], before[2][1])
    assert (c.codes[0, 6:9] == 0x5A).all() and (c.scales[0, 6:9] == 0x5A).all() and (c.ikeys[0, 6:9] == 0x5A).all()
