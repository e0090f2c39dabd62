"""Residual model 1 of the oracle (FP8): the channel scale normalised by the
prediction's exponent.  Pins: the table rule against its closed form for every
base bin and exponent, the base bins against a numpy evaluation of their
definition, exact round trips (escapes included), the coded size against the
model's ideal code length, and the gain over model 0 on the synthetic caches."""
import numpy as np
import pytest

from lossless_kv_cache_fp8_gb300 import synth


def test_table_rule_closed_form(orc):
    L = orc.lib()
    for base in range(256):
        for e in range(16):
            assert L.or_model1_table(base, e) == min(max(base - 4 * e, 0), 31), (base, e)


def test_bin_ext_extends_the_grid(orc):
    L = orc.lib()
    # inside the table grid the extended bin equals the ordinary one
    for q in [1 << 13, (1 << 13) + 1, 3 << 14, (1 << 21) - 1, 12345, 1 << 12]:
        assert L.or_bin_ext(q) == L.or_bin_from_q(q, 4)
    # above it, four bins per octave keep counting: bin = 4 (p - 13) + the two bits below the leading one
    for p in range(21, 60):
        for j in range(4):
            q = (4 + j) << (p - 2)
            assert L.or_bin_ext(q) == 4 * (p - 13) + j
            assert L.or_bin_ext(q + (1 << (p - 2)) - 1) == 4 * (p - 13) + j


def _ord(b):
    b = b.astype(np.int64)
    return np.where(b & 0x80, (~b) & 0xFF, b | 0x80)


def _small(n_layers=1, n_tokens=300, lane_syms=64, heads=2):
    return synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=n_layers, n_tokens=n_tokens,
                                                       lane_syms=lane_syms, n_heads=heads)


def test_base_bins_match_definition(orc):
    w = _small()
    t, p = synth.gen_kv(w, "cpu")
    tn, pn = t.numpy(), p.numpy()
    prm = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                        w.n_calib, model=1)
    bins, sums, _ = orc.calibrate(prm, tn.reshape(-1), pn.reshape(-1))
    nc = min(w.n_calib, w.n_tokens)
    r = np.abs(_ord(tn) - _ord(pn))[:, :, :, :nc, :]
    e = ((pn.astype(np.int64) >> 3) & 15)[:, :, :, :nc, :]
    S = (r << e).sum(axis=3).reshape(-1)                       # [slices*D]
    assert np.array_equal(np.minimum(S, 2 ** 32 - 1).astype(np.uint32), sums)
    q = (S << 16) // nc
    want = np.zeros_like(q)
    big = q >= (1 << 13)
    pw = np.array([int(v).bit_length() - 1 for v in q])
    want[big] = 4 * (pw[big] - 13) + ((q[big] >> (pw[big] - 2)) & 3)
    assert np.array_equal(bins.astype(np.int64), want)


@pytest.mark.parametrize("kw", [dict(), dict(n_tokens=333, lane_syms=32), dict(n_layers=2, heads=1)])
def test_round_trip_model1(orc, kw):
    w = _small(**kw)
    t, p = synth.gen_kv(w, "cpu")
    tn, pn = t.numpy().reshape(-1).copy(), p.numpy().reshape(-1).copy()
    # plant escapes: a few targets far from their predictions
    rng = np.random.default_rng(3)
    idx = rng.choice(tn.size, 40, replace=False)
    tn[idx] = (pn[idx].astype(np.int64) + 128 + rng.integers(0, 100, 40)).astype(np.uint8)
    prm = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                        w.n_calib, model=1)
    bins, _, _ = orc.calibrate(prm, tn, pn)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, tn, pn)
    assert st == orc.OK
    st, out = orc.decode(prm, fr, cum, bins, bs, offs, pn, np.uint8)
    assert st == orc.OK and np.array_equal(out, tn)


def test_model1_code_length_and_gain(orc):
    w = _small(n_layers=1, n_tokens=2048, lane_syms=256, heads=4)
    t, p = synth.gen_kv(w, "cpu")
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    sizes = {}
    for model in (0, 1):
        prm = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                            w.n_calib, model=model)
        bins, _, _ = orc.calibrate(prm, tn, pn)
        fr, cum = orc.build_tables(prm)
        st, bs, offs = orc.encode(prm, fr, cum, bins, tn, pn)
        assert st == orc.OK
        ideal = orc.shannon_bits(prm, fr, bins, tn, pn) / 8
        # rANS with 32-bit state stays within 1% (plus 4 state bytes per lane) of the model's code length
        lanes = offs.size - 1
        assert ideal <= bs.size <= ideal * 1.01 + 4 * lanes
        sizes[model] = bs.size
    assert sizes[1] < 0.9 * sizes[0]
