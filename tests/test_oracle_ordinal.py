"""Pins for the ordinal map and residual symbols (CPU only).

The ordinal is pinned against the float ordering of every FP8 / BF16 code,
computed by torch's own float decoding (an independent implementation): it must
be a bijection, monotone on non-NaN values, with -0 just below +0, and the
ordinal distance between two codes must equal their distance in the sorted list
of all codes.  Round trips over all 65,536 FP8 (target, pred) pairs and a mix of
BF16 pairs go through the whole oracle codec.
"""
import numpy as np
import pytest
import torch


def _float_values(width):
    codes = np.arange(1 << width, dtype=np.int64)
    if width == 8:
        t = torch.tensor(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    else:
        t = torch.tensor(codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64)
    return codes, t.numpy()


@pytest.mark.parametrize("width", [8, 16])
def test_ordinal_bijection_and_order(orc, width):
    codes, vals = _float_values(width)
    ords = np.array([orc.ordinal(int(c), width) for c in codes])
    assert sorted(ords.tolist()) == list(range(1 << width))          # bijection
    inv = np.array([orc.ordinal_inv(int(u), width) for u in ords])
    assert np.array_equal(inv, codes)
    ok = ~np.isnan(vals)
    # sorted order of all non-NaN codes by value, -0 below +0 (sign bit breaks ties)
    sign = (codes >> (width - 1)) & 1
    order = np.lexsort((1 - sign[ok], vals[ok]))
    ranked = codes[ok][order]
    o = ords[ranked]
    assert np.all(np.diff(o) == 1), "ordinals of the value-sorted codes are consecutive"
    # NaNs sit at the two ends
    nan_ords = sorted(ords[~ok].tolist())
    n_lo = sum(1 for u in nan_ords if u < o[0])
    assert n_lo + sum(1 for u in nan_ords if u > o[-1]) == len(nan_ords)
    top = 1 << (width - 1)
    assert orc.ordinal(top, width) + 1 == orc.ordinal(0, width)      # -0 just below +0


def test_fp8_all_pairs_roundtrip(orc):
    """every (target, pred) FP8 code pair through calibrate / tables / encode / decode"""
    t = np.repeat(np.arange(256, dtype=np.uint8), 256)
    p = np.tile(np.arange(256, dtype=np.uint8), 256)
    # cache [1][1][2][T=2048][16]: two heads, 2048 tokens x 16 channels
    prm = orc.kv_params(orc.FP8, 1, 1, 2, 16, 2048, lane_syms=64, n_calib=256)
    bins, _, _ = orc.calibrate(prm, t, p)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, t, p)
    assert st == orc.OK
    st, out = orc.decode(prm, fr, cum, bins, bs, offs, p, np.uint8)
    assert st == orc.OK
    assert np.array_equal(out, t)
    # escapes occurred (|r| > 127 exists among all pairs)
    _, syms, _ = orc.symbols(prm, bins, t, p)
    assert (syms == 255).sum() > 0 and (syms < 255).sum() > 0


def test_bf16_pairs_roundtrip(orc):
    rng = np.random.default_rng(7)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F7F, 0xFF7F, 0x0001,
                         0x8001, 0x3F80, 0xBF80], dtype=np.uint16)
    n = 1 * 2 * 2 * 2048 * 8
    t = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    p = t.astype(np.int64) + rng.integers(-300, 301, n)
    p = (p & 0xFFFF).astype(np.uint16)
    t[: specials.size * specials.size] = np.repeat(specials, specials.size)
    p[: specials.size * specials.size] = np.tile(specials, specials.size)
    prm = orc.kv_params(orc.BF16, 1, 2, 2, 8, 2048, lane_syms=128, n_calib=256)
    bins, _, _ = orc.calibrate(prm, t, p)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, t, p)
    assert st == orc.OK
    st, out = orc.decode(prm, fr, cum, bins, bs, offs, p, np.uint16)
    assert st == orc.OK and np.array_equal(out, t)
