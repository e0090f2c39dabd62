"""Checkerboard context of the oracle (coefficient rows split by token parity).
Pins: the context-shifted means against a numpy evaluation of their definition
(int64 matrix products, floor shifts, clamps; large values that hit every
clamp), exact fp32 means, a two-pass round trip (even rows decoded first, odd
rows' means rebuilt from them), and the gain of the context on the seeded
checkerboard data."""
import numpy as np
import torch

from lossless_kv_cache_fp8_gb300 import synth


def _numpy_ctx(V, U, s1, s2, qe, mo):
    V = np.clip(V.astype(np.int64), -8, 8); U = np.clip(U.astype(np.int64), -8, 8)
    n_o = mo.shape[0]
    right = np.zeros((n_o, qe.shape[1]), np.int64)
    n_r = min(n_o, qe.shape[0] - 1)
    right[:n_r] = qe[1:1 + n_r]
    x = np.clip(qe[:n_o].astype(np.int64) + right, -127, 127)
    g = np.clip(np.floor_divide(x @ V.T, 1 << s1), -127, 127)
    k = np.floor_divide(g @ U.T, 1 << s2)
    t = mo.astype(np.float32) * np.float32(16.0) + np.float32(0.5)
    mq = np.where(np.abs(t) < 2.0 ** 26, np.floor(t), 0).astype(np.int64)
    return np.clip(mq + k, -(2 ** 23 - 1), 2 ** 23 - 1)


def test_ctx_means_match_definition(orc):
    rng = np.random.default_rng(5)
    for (C, R, n_e, n_o) in [(48, 16, 7, 7), (40, 24, 9, 8), (16, 8, 1, 1)]:
        V = rng.integers(-8, 9, (R, C)).astype(np.int8)
        U = rng.integers(-8, 9, (C, R)).astype(np.int8)
        V[0, :3] = [127, -128, 9]          # entries outside [-8, 8] are used clamped
        U[1, :2] = [-100, 50]
        qe = rng.integers(-200, 201, (n_e, C)).astype(np.int16)
        qe[0, :5] = [32767, -32768, 127, -128, 0]
        mo = (rng.standard_normal((n_o, C)) * 50).astype(np.float32)
        mo[0, :3] = [1e9, -3.97, np.float32(0.03125)]
        for s1, s2 in [(6, 8), (0, 0), (3, 11)]:
            out = orc.ctx_means(V, U, s1, s2, qe, mo)
            want = _numpy_ctx(V, U, s1, s2, qe, mo)
            assert np.array_equal(out * np.float32(16.0), want.astype(np.float32))
            assert np.array_equal((out * 16).astype(np.int64), want)


def _coef_stream(orc, w, q, mu, beta):
    prm = orc.coef_params(q.shape[0], q.shape[1], w.lane_syms)
    bins, _, _ = orc.calibrate(prm, None, beta)
    fr, cum = orc.build_tables(prm)
    st, bs, offs = orc.encode(prm, fr, cum, bins, q.reshape(-1), mu.reshape(-1))
    assert st == orc.OK
    return prm, bins, fr, cum, bs, offs


def test_two_pass_round_trip_and_gain(orc):
    # the full-width map (2048 coefficients, rank 1024) on a few tokens
    w = synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=33, lane_syms=64)
    qe, qo, me, mo, beta, V, U = [x.numpy() for x in synth.gen_coef_checkerboard(w, "cpu")]
    s1, s2 = synth.CTX_SHIFT1, synth.CTX_SHIFT2
    # encode: even rows with their means, odd rows with the context-shifted means
    mo2 = orc.ctx_means(V, U, s1, s2, qe, mo)
    pe, be, fr, cum, bs_e, off_e = _coef_stream(orc, w, qe, me, beta)
    po, bo, _, _, bs_o, off_o = _coef_stream(orc, w, qo, mo2, beta)
    # decode: pass 1 (even rows), context from the decoded rows, pass 2 (odd rows)
    st, qe_d = orc.decode(pe, fr, cum, be, bs_e, off_e, me.reshape(-1), np.int16)
    assert st == orc.OK and np.array_equal(qe_d.reshape(qe.shape), qe)
    mo3 = orc.ctx_means(V, U, s1, s2, qe_d.reshape(qe.shape), mo)
    assert np.array_equal(mo3, mo2)
    st, qo_d = orc.decode(po, fr, cum, bo, bs_o, off_o, mo3.reshape(-1), np.int16)
    assert st == orc.OK and np.array_equal(qo_d.reshape(qo.shape), qo)
    # the context pays: odd rows cost fewer bytes than with the token-conditioned means alone
    _, _, _, _, bs_plain, _ = _coef_stream(orc, w, qo, mo, beta)
    assert bs_o.size < 0.9 * bs_plain.size
