"""Pins for calibration bins and the integer Laplace tables (CPU only).

* tau_q against exp(-1/(16 beta)) evaluated with mpmath (50 digits);
* masses against the closed-form Laplace cell integrals, within the rounding
  bound of the integer power chain; they add to exactly 2^32;
* frequencies: sum 4096, floor 1, mirror symmetry and monotone tails for f = 0;
* scale bins against an independent integer formulation (octave from
  bit_length, linear sub-bin from a division) and against sums of |r| computed
  from value-sorted code ranks (no ordinal formula involved).
"""
import mpmath as mp
import numpy as np
import pytest
import torch

mp.mp.dps = 50


def beta_exact(b, sub):
    e, j = divmod(b, sub)
    return mp.mpf(2) ** (e - 3) * (1 + (mp.mpf(j) + mp.mpf(1) / 2) / sub)


@pytest.mark.parametrize("sub", [4, 8])
def test_beta_grid(orc, sub):
    for b in range(8 * sub):
        assert mp.mpf(orc.beta_q(b, sub)) / 65536 == beta_exact(b, sub)


@pytest.mark.parametrize("sub", [4, 8])
def test_tau_against_mpmath(orc, sub):
    for b in range(8 * sub):
        beta = mp.mpf(orc.beta_q(b, sub)) / 65536
        tau = mp.exp(-1 / (16 * beta))
        got = mp.mpf(orc.tau_q(orc.beta_q(b, sub))) / 2 ** 32
        assert abs(got - tau) <= mp.mpf(64) / 2 ** 32, (b, got, tau)


def laplace_cell(beta, lo, hi):
    """P(lo <= Y < hi) for Y ~ Laplace(0, beta); lo/hi may be +-inf"""
    def F(y):
        if y == mp.inf:
            return mp.mpf(1)
        if y == -mp.inf:
            return mp.mpf(0)
        return mp.exp(y / beta) / 2 if y < 0 else 1 - mp.exp(-y / beta) / 2
    return F(hi) - F(lo)


@pytest.mark.parametrize("sub,b,f", [(4, 0, 0), (4, 7, 0), (4, 16, 0), (4, 31, 0),
                                     (8, 0, 3), (8, 33, 8), (8, 63, 15), (8, 40, 1)])
def test_masses_closed_form(orc, sub, b, f):
    m = orc.masses(b, sub, f)
    assert int(m.astype(object).sum()) == 1 << 32          # telescoping: exact
    beta = mp.mpf(orc.beta_q(b, sub)) / 65536
    mu = mp.mpf(f) / 16
    # rounding of 2055 chained Q32 multiplies and of tau: a few 1e-7 at most
    tol = mp.mpf("2e-6")
    for i in range(255):
        s = i - 127
        want = laplace_cell(beta, s - mp.mpf(1) / 2 - mu, s + mp.mpf(1) / 2 - mu)
        assert abs(mp.mpf(int(m[i])) / 2 ** 32 - want) <= tol, (i, m[i], want)
    esc = laplace_cell(beta, -mp.inf, -127 - mp.mpf(1) / 2 - mu) + \
        laplace_cell(beta, 127 + mp.mpf(1) / 2 - mu, mp.inf)
    assert abs(mp.mpf(int(m[255])) / 2 ** 32 - esc) <= tol


@pytest.mark.parametrize("sub", [4, 8])
def test_frequency_invariants(orc, sub):
    fs = range(16) if sub == 8 else [0]
    for b in range(8 * sub):
        for f in fs:
            fr, cum = orc.build_table(b, sub, f)
            fr = fr.astype(np.int64)
            assert fr.sum() == 4096 and fr.min() >= 1
            assert cum[0] == 0 and cum[256] == 4096
            assert np.array_equal(np.diff(cum.astype(np.int64)), fr)
            m = orc.masses(b, sub, f).astype(np.float64) / 2 ** 32
            # quota check: every frequency is within one unit of 1 + m*3840
            assert np.all(np.abs(fr - (1 + m * 3840)) < 1.0 + 1e-9)
            if f == 0:
                for s in range(1, 128):
                    d = fr[127 - s] - fr[127 + s]
                    assert d in (0, 1), (b, s, d)      # mirror masses, ties to lower index
                for side in (fr[127::-1], fr[127:255]):
                    assert np.all(np.diff(side) <= 0)  # non-increasing away from 0


def test_cross_entropy_close_to_model(orc):
    """the integer table costs at most ~0.1 bit/symbol over the model's own entropy
    (the floor of 1 for 255 tail symbols costs ~0.09 bit at low entropy)"""
    for sub in (4, 8):
        for b in range(8 * sub):
            m = orc.masses(b, sub, 0).astype(np.float64) / 2 ** 32
            fr, _ = orc.build_table(b, sub, 0)
            nz = m > 0
            H = -(m[nz] * np.log2(m[nz])).sum()
            ce = -(m * np.log2(fr / 4096.0)).sum()
            assert ce - H < 0.1, (sub, b, ce - H)


@pytest.mark.parametrize("sub", [4, 8])
def test_bin_from_q(orc, sub):
    nb = 8 * sub
    qs = list(range(0, 1 << 14, 7)) + list(range((1 << 13) - 5, (1 << 13) + 5)) + \
        [int(x) for x in np.unique(np.geomspace(1 << 13, 1 << 22, 4000).astype(np.int64))] + \
        [(1 << 21) - 1, 1 << 21, (1 << 40)]
    for q in qs:
        if q < 1 << 13:
            want = 0
        elif q >= 1 << 21:
            want = nb - 1
        else:
            p = q.bit_length() - 1
            want = sub * (p - 13) + ((q - (1 << p)) * sub) // (1 << p)
        assert orc.bin_from_q(q, sub) == want, q


def _rank_table(width):
    """ordinal distance from value ranks: position of each code in the value-sorted
    list of all codes (NaN codes placed by the convention: sign-set NaNs first)."""
    codes = np.arange(1 << width, dtype=np.int64)
    if width == 8:
        v = torch.tensor(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        v = torch.tensor(codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    sign = (codes >> (width - 1)) & 1
    nan = np.isnan(v)
    # key: negative NaNs lowest, then values (with -0 < +0), then positive NaNs; within
    # NaNs of one sign, order by magnitude bits (more negative first for sign-set ones)
    mag = codes & ((1 << (width - 1)) - 1)
    grp = np.where(nan & (sign == 1), 0, np.where(nan, 2, 1))
    sub_key = np.where(nan & (sign == 1), -mag, np.where(nan, mag, 0))
    vv = np.where(nan, 0.0, v)
    order = np.lexsort((sub_key, 1 - sign, vv, grp))
    rank = np.empty_like(codes)
    rank[order] = np.arange(codes.size)
    return rank


@pytest.mark.parametrize("dtype,width", [(1, 8), (2, 16)])
def test_calibration_against_ranks(orc, dtype, width):
    rng = np.random.default_rng(11)
    L, KV, H, T, D = 2, 2, 1, 300, 16
    n = L * KV * H * T * D
    if width == 8:
        t = rng.integers(0, 256, n).astype(np.uint8)
        p = t.astype(np.int64) + rng.integers(-3, 4, n) * (rng.random(n) < 0.5)
        p = np.clip(p, 0, 255).astype(np.uint8)
    else:
        t = rng.integers(0, 1 << 16, n).astype(np.uint16)
        p = ((t.astype(np.int64) + rng.integers(-40, 41, n)) & 0xFFFF).astype(np.uint16)
    prm = orc.kv_params(dtype, L, KV, H, D, T, lane_syms=64, n_calib=256)
    bins, sums, hist = orc.calibrate(prm, t, p, want_sum=True, want_hist=True)
    rank = _rank_table(width)
    r = rank[t.astype(np.int64)] - rank[p.astype(np.int64)]
    r = r.reshape(L * KV * H, T, D)[:, :256, :]
    S = np.abs(r).sum(axis=1).reshape(-1)
    assert np.array_equal(sums.astype(np.int64), S)
    for c in range(S.size):
        q = (int(S[c]) << 16) // 256
        assert bins[c] == orc.bin_from_q(q, 4)
    assert np.all(hist.sum(axis=1) == 256)


def test_calibration_uses_first_tokens_only(orc):
    rng = np.random.default_rng(3)
    L, KV, H, T, D = 1, 2, 2, 600, 16
    n = L * KV * H * T * D
    t = rng.integers(0, 256, n).astype(np.uint8)
    p = np.clip(t.astype(np.int64) + rng.integers(-2, 3, n), 0, 255).astype(np.uint8)
    prm = orc.kv_params(1, L, KV, H, D, T, lane_syms=64, n_calib=256)
    b1, _, _ = orc.calibrate(prm, t, p)
    t2 = t.reshape(-1, T, D).copy()
    t2[:, 256:, :] = rng.integers(0, 256, t2[:, 256:, :].shape)
    b2, _, _ = orc.calibrate(prm, t2.reshape(-1), p)
    assert np.array_equal(b1, b2)


def test_coef_skip_rule(orc):
    beta = np.array([0.0, 0.049999, np.float32(0.05), 0.0625, 0.2, 31.9, 32.0, 1e9, np.nan, -1.0],
                    dtype=np.float32)
    prm = orc.coef_params(4, beta.size, lane_syms=8)
    bins, _, _ = orc.calibrate(prm, None, beta)
    assert bins.tolist()[:3] == [0xFF, 0xFF, 0]
    assert bins[3] == 0                       # beta below 1/8: first bin
    assert bins[6] == 63 and bins[7] == 63
    assert bins[8] == 0xFF and bins[9] == 0xFF
    q = int(np.floor(np.float32(0.2) * np.float32(65536)))
    assert bins[4] == orc.bin_from_q(q, 8)


@pytest.mark.parametrize("sub", [4, 8])
def test_power_chain_rounding_bound(orc, sub):
    """P[n] = round(P[n-1] tau): against the exact power of the integer tau_q the error
    obeys |e_n| <= tau |e_{n-1}| + 1/2, hence |e_n| <= min(n/2, 1/(2(1 - tau)));
    a truncating chain drifts to about twice that."""
    for b in range(0, 8 * sub, 3):
        tq = orc.tau_q(orc.beta_q(b, sub))
        P = orc.power_chain(tq)
        tau = mp.mpf(tq) / 2 ** 32
        bound = mp.mpf(1) / (2 * (1 - tau))
        x = mp.mpf(2) ** 32
        for n in range(1, 2056):
            x *= tau
            assert abs(mp.mpf(int(P[n])) - x) <= min(mp.mpf(n) / 2, bound) + mp.mpf("1e-9"), (b, n)


def test_coef_mean_quantisation(orc):
    """table choice: mu rounded to the nearest 1/16 (ties upward), integer part m
    shifts the residual, fraction f picks the table (16*bin + f)"""
    from fractions import Fraction
    mus = np.array([0.0, 0.03125, -0.03125, 0.0624, 0.0938, -0.0313, 1.5, -1.5, 2.96875,
                    -2.96875, 100.03, -7.99, 0.4999, -0.4999], dtype=np.float32)
    T, Cc = 1, mus.size
    beta = np.full(Cc, 1.0, np.float32)
    prm = orc.coef_params(T, Cc, lane_syms=8)
    bins, _, _ = orc.calibrate(prm, None, beta)
    q = np.full(Cc, 3, np.int16)
    tables, syms, _ = orc.symbols(prm, bins, q, mus)
    for i, mu in enumerate(mus):
        mq = Fraction(float(mu)) * 16
        n = int(np.floor(mq + Fraction(1, 2)))          # nearest, ties up
        m, f = n // 16, n % 16
        assert int(tables[i]) == 16 * int(bins[i]) + f, (mu, tables[i], f)
        assert int(syms[i]) == 3 - m + 127, (mu, syms[i], m)


@pytest.mark.parametrize("width", [8, 16])
def test_symbols_from_ranks(orc, width):
    rng = np.random.default_rng(5)
    n = 64 * 16
    hi = 1 << width
    t = rng.integers(0, hi, n)
    p = np.where(rng.random(n) < 0.7, (t + rng.integers(-130, 131, n)) % hi, rng.integers(0, hi, n))
    dt = np.uint8 if width == 8 else np.uint16
    prm = orc.kv_params(1 if width == 8 else 2, 1, 1, 1, 16, 64, lane_syms=16, n_calib=16)
    t, p = t.astype(dt), p.astype(dt)
    bins, _, _ = orc.calibrate(prm, t, p)
    _, syms, raw = orc.symbols(prm, bins, t, p)
    rank = _rank_table(width)
    r = rank[t.astype(np.int64)] - rank[p.astype(np.int64)]
    direct = np.abs(r) <= 127
    assert np.array_equal(syms[direct], r[direct] + 127)
    assert np.all(syms[~direct] == 255)
    assert np.array_equal(raw[~direct].astype(np.int64), r[~direct] % hi)
