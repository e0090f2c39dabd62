"""Independent pins for two oracle steps that its round trips cannot fix (CPU only).

1. Largest-remainder frequencies ([DCKV] "how it differs": Laplace integrated
   over the quantisation cells, quantised to 12-bit frequencies).  Checked two
   ways that do not rerun the oracle's allocation loop:
   * the defining Hamilton property on every KV table and every COEF table:
     with the oracle's Q32 masses (themselves pinned against closed forms in
     test_oracle_tables.py), each frequency is 1 + floor(3840 m / 2^32) plus a
     bonus of 0 or 1, the bonuses fill the deficit to 4096, and every symbol
     with a bonus has a larger remainder than every symbol without one (equal
     remainders: the lower symbol index first);
   * hand-derived tables (tests/golden/laplace_tables.txt): bins 0, 15 and 31
     of the KV grid and one mean-shifted coefficient table, worked out from
     the closed-form Laplace cell masses.
2. Lane layout, against the stream format stated in include/skv.h: lane l of
   a chunk owns the 16-byte groups whose chunk-local index is l mod 32; lanes
   are stored in the order chunk*32 + l; lane_offsets is the byte prefix of the
   lane lengths.  A cache whose prediction equals the target except at one
   position must change exactly one lane: the one those words name.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "laplace_tables.txt")


def _hamilton_ok(fr, m):
    """fr: 256 frequencies, m: 256 Q32 masses (python ints).  True when fr is
    the largest-remainder allocation of 3840 units over the floors + 1."""
    scaled = [mi * 3840 for mi in m]
    base = [1 + (s >> 32) for s in scaled]
    rem = [s & 0xFFFFFFFF for s in scaled]
    bonus = [int(f) - b for f, b in zip(fr, base)]
    if any(b not in (0, 1) for b in bonus):
        return False
    if sum(base) + sum(bonus) != 4096:
        return False
    # priority: larger remainder first, then the lower index
    key = [r * 256 + (255 - i) for i, r in enumerate(rem)]
    got = [key[i] for i in range(256) if bonus[i]]
    not_got = [key[i] for i in range(256) if not bonus[i]]
    return not got or not not_got or min(got) > max(not_got)


@pytest.mark.parametrize("sub", [4, 8])
def test_largest_remainder_is_hamilton(orc, sub):
    fs = range(16) if sub == 8 else [0]
    n_with_deficit = 0
    for b in range(8 * sub):
        for f in fs:
            fr, _ = orc.build_table(b, sub, f)
            m = [int(v) for v in orc.masses(b, sub, f)]
            assert _hamilton_ok(fr, m), (sub, b, f)
            n_with_deficit += int(sum(1 + ((mi * 3840) >> 32) for mi in m) < 4096)
    assert n_with_deficit > 0   # the bonus step is exercised


def test_hamilton_check_rejects_other_allocations(orc):
    """The property check itself fails for the plausible wrong rules: units to
    the smallest remainders, in index order, or ties to the higher index."""
    m = [int(v) for v in orc.masses(15, 4, 0)]
    scaled = [mi * 3840 for mi in m]
    base = np.array([1 + (s >> 32) for s in scaled])
    rem = np.array([s & 0xFFFFFFFF for s in scaled], dtype=np.uint64)
    d = 4096 - int(base.sum())
    assert d > 0
    idx = np.arange(256)
    for order in (np.lexsort((idx, rem)),                   # smallest remainders first
                  idx,                                      # index order
                  np.lexsort((-idx, -rem.astype(np.int64)))):  # ties to the higher index
        fr = base.copy()
        fr[order[:d]] += 1
        assert not _hamilton_ok(fr, m)


def _read_golden():
    tables, cur = [], None
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "table":
                kv = dict(t.split("=") for t in tok[2:])
                cur = dict(kind=tok[1], sub=int(kv["sub"]), bin=int(kv["bin"]), f=int(kv["f"]), sym={})
            elif tok[0] == "deficit":
                cur["deficit"] = int(tok[1])
            elif tok[0] == "bonus":
                cur["bonus"] = tok[1:]
            elif tok[0] == "sym":
                i = 255 if tok[1] == "esc" else int(tok[1]) + 127
                cur["sym"][i] = int(tok[3])
            elif tok[0] == "end":
                tables.append(cur)
    return tables


def test_golden_tables_hand_derived(orc):
    tables = _read_golden()
    assert [(t["sub"], t["bin"], t["f"]) for t in tables] == [(4, 0, 0), (4, 15, 0), (4, 31, 0), (8, 24, 4)]
    for t in tables:
        fr, cum = orc.build_table(t["bin"], t["sub"], t["f"])
        want = np.ones(256, np.int64)
        for i, v in t["sym"].items():
            want[i] = v
        assert want.sum() == 4096
        assert np.array_equal(fr.astype(np.int64), want), (t["sub"], t["bin"], t["f"])
        assert np.array_equal(np.cumsum(np.concatenate([[0], want])), cum.astype(np.int64))


# --- lane layout -----------------------------------------------------------------------------
def _lane_lengths(offs):
    o = offs.astype(np.int64)
    return np.diff(o)


def _layout_case(orc, dtype, n_heads, n_tokens, head_dim, K, positions):
    """Encode a cache with prediction == target, then with one position
    changed, for each position; return what changed."""
    width = 8 if dtype == orc.FP8 else 16
    prm = orc.kv_params(dtype, 1, 2, n_heads, head_dim, n_tokens, K, 16)
    g = orc.geometry(prm)
    n = g["n_slices"] * g["slice_positions"]
    rng = np.random.default_rng(7)
    np_dt = np.uint8 if width == 8 else np.uint16
    # finite values of moderate magnitude (no NaN patterns)
    tgt = rng.integers(0, 0x30 if width == 8 else 0x3000, n).astype(np_dt)
    pred = tgt.copy()
    bins = np.zeros(g["n_channels"], np.uint8)      # every channel on the sharpest table
    fr, cum = orc.build_tables(prm)
    st, bs0, off0 = orc.encode(prm, fr, cum, bins, tgt, pred)
    assert st == orc.OK
    len0 = _lane_lengths(off0)
    assert off0[0] == 0 and int(off0[-1]) == bs0.size and np.all(len0 >= 4)
    G = 16 if width == 8 else 8
    chunk_pos = 32 * K
    for P in positions:
        t2 = tgt.copy()
        t2[P] = t2[P] ^ (0x40 if width == 8 else 0x4000)   # large residual: an escape
        st, bs1, off1 = orc.encode(prm, fr, cum, bins, t2, pred)
        assert st == orc.OK
        len1 = _lane_lengths(off1)
        # the lane the header's words name
        sl, local = divmod(P, g["slice_positions"])
        c_in, j = divmod(local, chunk_pos)
        lane = (sl * g["chunks_per_slice"] + c_in) * 32 + (j // G) % 32
        changed = np.nonzero(len1 != len0)[0]
        assert list(changed) == [lane], (P, lane, changed)
        assert len1[lane] > len0[lane]
        # lanes before it keep their bytes and offsets; lanes after it move by
        # the growth and keep their bytes (lanes concatenated in lane order)
        a = int(off0[lane])
        delta = int(len1[lane] - len0[lane])
        assert np.array_equal(off1[: lane + 1], off0[: lane + 1])
        assert np.array_equal(off1[lane + 1:].astype(np.int64), off0[lane + 1:].astype(np.int64) + delta)
        assert np.array_equal(bs1[:a], bs0[:a])
        b0 = int(off0[lane + 1])
        assert np.array_equal(bs1[b0 + delta:], bs0[b0:])


def test_lane_layout_fp8(orc):
    # 2 slices of 40 x 128 positions, K = 64: chunks of 2048, the last one of each slice ragged
    n = 2 * 40 * 128
    pos = [0, 15, 16, 31 * 16, 32 * 16, 32 * 16 + 5, 2047, 2048, 2048 + 33 * 16 + 1,
           4096 + 7, 5119, 5120, 5120 + 4096 + 100, n - 1]
    _layout_case(orc, orc.FP8, 1, 40, 128, 64, pos)


def test_lane_layout_bf16(orc):
    # 4 heads of 24 tokens x 64 channels, K = 32: chunks of 1024 positions, 8-value groups
    n = 2 * 4 * 24 * 64
    pos = [0, 7, 8, 31 * 8, 32 * 8 + 3, 1023, 1024, 1536 + 9, 3 * 1536 + 1024 + 64 + 2, n - 1]
    _layout_case(orc, orc.BF16, 4, 24, 64, 32, pos)
