"""Whole-codec pins for the oracle (CPU only): lossless round trips on small
versions of every workload and on ragged / degenerate shapes, the coded length
against the Shannon sum, chunk-level calls against the whole-stream calls, and
corruption detection."""
import numpy as np
import pytest

from lossless_kv_cache_fp8_gb300 import synth


def small(name, **kw):
    w = synth.WORKLOADS[name]
    return w.scaled(**kw)


def oracle_params(orc, w):
    if w.dtype == synth.COEF:
        return orc.coef_params(w.n_tokens, w.n_coef, w.lane_syms)
    return orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens,
                         w.lane_syms, w.n_calib)


def gen_np(w):
    t, p, c = synth.gen_workload(w, "cpu")
    if w.dtype == synth.COEF:
        return t.numpy().reshape(-1), p.numpy().reshape(-1), c.numpy()
    to = lambda x: x.numpy().reshape(-1).view(np.uint8 if w.dtype == synth.FP8 else np.uint16)
    return to(t), to(p), to(c)


def roundtrip(orc, w):
    prm = oracle_params(orc, w)
    t, p, c = gen_np(w)
    bins, _, _ = orc.calibrate(prm, None if w.dtype == synth.COEF else t, c)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, t, p)
    assert st == orc.OK
    out_dt = np.int16 if w.dtype == synth.COEF else t.dtype
    st, out = orc.decode(prm, fr, cum, bins, bs, offs, p, out_dt)
    assert st == orc.OK
    assert np.array_equal(out.view(out_dt), t.view(out_dt))
    return prm, t, p, bins, fr, cum, bs, offs


SMALL = [
    small("qwen3-0.6b-1k-fp8", n_layers=2, n_tokens=512),
    small("qwen3-0.6b-8k-bf16", n_layers=1, n_tokens=384),
    small("qwen3-8b-32k-fp8", n_layers=1, n_heads=2, n_tokens=1024, lane_syms=256),
    small("hybrid-coef-32k-x2048", n_tokens=64, n_coef=256, lane_syms=64),
    # ragged: tokens not a multiple of the chunk, short calibration, odd lane sizes
    small("qwen3-0.6b-1k-fp8", n_layers=1, n_heads=3, n_tokens=77, head_dim=32, lane_syms=48),
    small("qwen3-0.6b-8k-bf16", n_layers=1, n_heads=1, n_tokens=1, head_dim=16, lane_syms=8),
    small("hybrid-coef-32k-x2048", n_tokens=7, n_coef=37, lane_syms=24),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"{w.name}-T{w.n_tokens}-K{w.lane_syms}")
def test_roundtrip_and_shannon(orc, w):
    prm, t, p, bins, fr, cum, bs, offs = roundtrip(orc, w)
    g = orc.geometry(prm)
    assert offs.size == g["n_lanes"] + 1 and int(offs[-1]) == bs.size
    assert np.all(np.diff(offs.astype(np.int64)) >= 4) and np.all(offs % 2 == 0)
    bits = orc.shannon_bits(prm, fr, bins, t, p)
    assert 8 * bs.size <= 1.005 * bits + 32 * g["n_lanes"] + 16 * g["n_lanes"]


def test_chunk_calls_match_stream(orc):
    w = SMALL[4]
    prm, t, p, bins, fr, cum, bs, offs = roundtrip(orc, w)
    g = orc.geometry(prm)
    sp = g["slice_positions"]
    words = bs.view(np.uint16)
    for chunk in range(g["n_chunks"]):
        sl, k = divmod(chunk, g["chunks_per_slice"])
        first = sl * sp + k * 32 * w.lane_syms
        n_pos = min(32 * w.lane_syms, sp - k * 32 * w.lane_syms)
        cw, lw = orc.encode_chunk(prm, chunk, fr, cum, bins, t[first:first + n_pos], p[first:first + n_pos])
        a, b = int(offs[32 * chunk]) // 2, int(offs[32 * chunk + 32]) // 2
        assert np.array_equal(cw, words[a:b])
        assert np.array_equal(lw.astype(np.int64), np.diff(offs[32 * chunk:32 * chunk + 33].astype(np.int64)) // 2)
        st, out = orc.decode_chunk(prm, chunk, fr, cum, bins, cw, lw, p[first:first + n_pos], n_pos, t.dtype)
        assert st == orc.OK and np.array_equal(out, t[first:first + n_pos])


def test_empty_stream(orc):
    prm = orc.kv_params(1, 1, 2, 1, 16, 0, lane_syms=16)
    g = orc.geometry(prm)
    assert g["n_chunks"] == 0 and g["n_lanes"] == 0
    t = np.zeros(1, np.uint8)
    bins, _, _ = orc.calibrate(prm, t, t)
    assert np.all(bins == 0)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, t, t)
    assert st == orc.OK and bs.size == 0 and offs.tolist() == [0]


def test_identical_prediction_is_cheap(orc):
    """target == prediction: every residual is 0, the stream is near the floor"""
    w = small("qwen3-0.6b-1k-fp8", n_layers=1, n_tokens=512)
    prm = oracle_params(orc, w)
    t, _, _ = gen_np(w)
    bins, _, _ = orc.calibrate(prm, t, t)
    assert np.all(bins == 0)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, t, t)
    assert st == orc.OK
    st, out = orc.decode(prm, fr, cum, bins, bs, offs, t, np.uint8)
    assert st == orc.OK and np.array_equal(out, t)
    p0 = fr[0, 127] / 4096.0
    n_lanes = orc.geometry(prm)["n_lanes"]
    assert 8 * bs.size <= 1.005 * (-np.log2(p0) * t.size) + 48 * n_lanes


def test_corruption_detected(orc):
    w = SMALL[0]
    prm, t, p, bins, fr, cum, bs, offs = roundtrip(orc, w)
    # truncated stream: offsets no longer end at n_bytes
    st, _ = orc.decode(prm, fr, cum, bins, bs[:-2], offs, p, np.uint8)
    assert st == orc.ERR_CORRUPT
    # a lane's state words damaged: its final state cannot return to 2^16
    bad = bs.copy()
    a = int(offs[5])
    bad[a + 1] ^= 0x40
    st, out = orc.decode(prm, fr, cum, bins, bad, offs, p, np.uint8)
    assert st == orc.ERR_CORRUPT
    # offsets out of order
    o2 = offs.copy()
    o2[3], o2[4] = o2[4], o2[3]
    st, _ = orc.decode(prm, fr, cum, bins, bs, o2, p, np.uint8)
    assert st == orc.ERR_CORRUPT


def test_capacity_reported(orc):
    w = SMALL[0]
    prm = oracle_params(orc, w)
    t, p, c = gen_np(w)
    bins, _, _ = orc.calibrate(prm, t, c)
    fr, cum = orc.build_tables(prm)
    st, _, _ = orc.encode(prm, fr, cum, bins, t, p, cap_bytes=100)
    assert st == orc.ERR_CAPACITY


def test_param_checks(orc):
    assert orc.check_params(orc.kv_params(1, 1, 2, 1, 24, 10, lane_syms=16)) == orc.ERR_ARG   # head_dim % 16
    assert orc.check_params(orc.kv_params(1, 1, 2, 1, 16, 10, lane_syms=24)) == orc.ERR_ARG   # K % 16
    assert orc.check_params(orc.kv_params(2, 1, 2, 1, 8, 10, lane_syms=24)) == orc.OK          # bf16: groups of 8
    assert orc.check_params(orc.kv_params(9, 1, 2, 1, 16, 10, lane_syms=16)) == orc.ERR_ARG
