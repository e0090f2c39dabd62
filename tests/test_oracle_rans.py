"""Pins for the oracle's rANS coder (CPU only).

* hand-worked examples (tests/golden/rans_hand_examples.txt, derived by hand);
* brute force: every sequence of length <= 4 over 3- and 4-symbol toy tables
  round-trips and ends in the initial state;
* random long sequences over real tables round-trip and cost at most 0.5% above
  the Shannon sum -sum log2 p plus the 32-bit final state.
"""
import itertools
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rans_hand_examples.txt")


def _parse_golden():
    ex, cur = [], None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "example":
            cur = {"name": vals[0]}
        elif key == "end":
            ex.append(cur)
            cur = None
        else:
            cur[key] = vals
    return ex


def _table(e):
    if e["freq"] == ["uniform16"]:
        return [16] * 256, [16 * i for i in range(256)]
    fr = [int(v, 0) for v in e["freq"]]
    return fr, [int(v, 0) for v in e["cum"]]


@pytest.mark.parametrize("ex", _parse_golden(), ids=lambda e: e["name"])
def test_hand_examples(orc, ex):
    pb = int(ex["prob_bits"][0])
    fr, cum = _table(ex)
    syms = [int(v, 0) for v in ex["symbols"]]
    want = [int(v, 0) for v in ex["stream"]]
    got = orc.rans_encode(pb, fr, cum, syms)
    assert [int(w) for w in got] == want
    st, dec = orc.rans_decode(pb, fr, cum, np.array(want, np.uint16), len(syms))
    assert st == orc.OK
    assert [int(s) for s in dec] == syms


TOYS = [
    (2, [2, 1, 1]),              # M = 4
    (3, [5, 2, 1]),              # M = 8
    (3, [1, 1, 3, 3]),
    (12, [4000, 64, 31, 1]),     # extreme skew, renormalises often
]


@pytest.mark.parametrize("pb,fr", TOYS)
def test_bruteforce_short_sequences(orc, pb, fr):
    cum = np.concatenate([[0], np.cumsum(fr)[:-1]])
    assert sum(fr) == 1 << pb
    for n in range(0, 5):
        for seq in itertools.product(range(len(fr)), repeat=n):
            words = orc.rans_encode(pb, fr, cum, list(seq))
            st, dec = orc.rans_decode(pb, fr, cum, words, n)
            assert st == orc.OK, (seq, words)
            assert list(dec) == list(seq)


def test_decode_detects_wrong_length(orc):
    fr, cum = [2, 1, 1], [0, 2, 3]
    words = orc.rans_encode(2, fr, cum, [0, 1, 2, 1, 0])
    st, _ = orc.rans_decode(2, fr, cum, words, 4)      # one symbol short: state != L
    assert st == orc.ERR_CORRUPT
    st, _ = orc.rans_decode(2, fr, cum, words[:1], 5)  # truncated stream
    assert st == orc.ERR_CORRUPT


@pytest.mark.parametrize("sub,b,f", [(4, 0, 0), (4, 9, 0), (4, 31, 0), (8, 17, 5), (8, 63, 15)])
def test_random_long_sequences_shannon(orc, sub, b, f):
    fr, cum = orc.build_table(b, sub, f)
    fr = fr.astype(np.int64)
    p = fr / 4096.0
    rng = np.random.default_rng(1234 + 64 * sub + b + f)
    n = 100_000
    syms = rng.choice(256, size=n, p=p)
    words = orc.rans_encode(12, fr, cum[:256], syms)
    st, dec = orc.rans_decode(12, fr, cum[:256], words, n)
    assert st == orc.OK
    assert np.array_equal(dec, syms)
    shannon = float(-np.log2(p[syms]).sum())
    coded = 16.0 * len(words)
    # rANS with L/M = 16 loses ~1e-3 bit/symbol; 0.5% plus the final state and one word
    assert coded <= 1.005 * shannon + 32 + 16, (coded, shannon)
