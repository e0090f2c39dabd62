"""Mutation check of the oracle's pins (CPU only; run by hand, not collected by pytest).

Each mutation plants one plausible mistake in a temporary copy of
oracle/skv_oracle.c (a dropped term, a wrong sign, bound or index, a swapped
operand), builds it with gcc and runs the CPU pin tests against that build
(SKV_ORACLE_LIB points the oracle wrapper at it).  Every mutation must make at
least one pin fail; the script prints which test caught it and exits non-zero
if any mutation survives.

    python tests/oracle_mutations.py            # all mutations
    python tests/oracle_mutations.py tau-sign   # one by name
"""
import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "skv_oracle.c")
PIN_TESTS = ["tests/test_oracle_pins.py", "tests/test_oracle_rans.py", "tests/test_oracle_tables.py",
             "tests/test_oracle_ordinal.py", "tests/test_oracle_codec.py", "tests/test_oracle_model1.py",
             "tests/test_oracle_checkerboard.py"]

# name -> (text in the source, replacement); each text occurs exactly once
MUTATIONS = {
    "ordinal-drops-top": ("  return bits | top;", "  return bits;"),
    "ordinal-inverse-keeps-top": ("if (u & top) return u & ~top;", "if (u & top) return u;"),
    "bin-octave-offset": ("return sub * (pw - 13u) + (uint32_t)((q >> (pw - sb)) & (sub - 1u));",
                          "return sub * (pw - 12u) + (uint32_t)((q >> (pw - sb)) & (sub - 1u));"),
    "bin-sub-bits": ("return sub * (pw - 13u) + (uint32_t)((q >> (pw - sb)) & (sub - 1u));",
                     "return sub * (pw - 13u) + (uint32_t)((q >> (pw - sb - 1u)) & (sub - 1u));"),
    "beta-lower-edge": ("(2ull * sub + 2ull * j + 1ull)", "(2ull * sub + 2ull * j)"),
    "tau-sign": ("tau += (n & 1) ? -(int64_t)a : (int64_t)a;", "tau += (n & 1) ? (int64_t)a : -(int64_t)a;"),
    "tau-x-scale": ("uint64_t x_q = ((1ull << 44) + (beta_q >> 1)) / beta_q;",
                    "uint64_t x_q = ((1ull << 43) + (beta_q >> 1)) / beta_q;"),
    "chain-truncates": ("P[n] = (P[n - 1] * tau_q + (1ull << 31)) >> 32;", "P[n] = (P[n - 1] * tau_q) >> 32;"),
    "cdf-halving": ("if (n < 0) return P[-n] >> 1;", "if (n < 0) return P[-n] >> 2;"),
    "cell-width": ("m[i] = cdf16(P, 16 * s + 8 - (int64_t)f) - cdf16(P, 16 * s - 8 - (int64_t)f);",
                   "m[i] = cdf16(P, 16 * s + 7 - (int64_t)f) - cdf16(P, 16 * s - 8 - (int64_t)f);"),
    "mean-shift-sign": ("m[i] = cdf16(P, 16 * s + 8 - (int64_t)f) - cdf16(P, 16 * s - 8 - (int64_t)f);",
                        "m[i] = cdf16(P, 16 * s + 8 + (int64_t)f) - cdf16(P, 16 * s - 8 + (int64_t)f);"),
    "remainder-smallest": ("if (best == NSYM || rem[i] > rem[best]) best = i;",
                           "if (best == NSYM || rem[i] < rem[best]) best = i;"),
    "remainder-ties-high": ("if (best == NSYM || rem[i] > rem[best]) best = i;",
                            "if (best == NSYM || rem[i] >= rem[best]) best = i;"),
    "remainder-index-order": ("if (best == NSYM || rem[i] > rem[best]) best = i;", "if (best == NSYM) best = i;"),
    "freq-scale": ("uint64_t scaled = m[i] * (uint64_t)(PROB_SCALE - NSYM);",
                   "uint64_t scaled = m[i] * (uint64_t)(PROB_SCALE - NSYM - 1);"),
    "escape-bound": ("if (r >= -RMAX && r <= RMAX) {", "if (r >= -RMAX && r < RMAX) {"),
    "escape-raw-width": ("o->raw = (uint32_t)((uint64_t)r & ((1ull << width) - 1ull));",
                         "o->raw = (uint32_t)((uint64_t)r & ((1ull << (width - 1u)) - 1ull));"),
    "raw-byte-order": ("enc_step(&e, PROB_BITS, 16u, 16u * ((s.raw >> (8u * b)) & 0xFFu));",
                       "enc_step(&e, PROB_BITS, 16u, 16u * ((s.raw >> (8u * (rb - 1u - b))) & 0xFFu));"),
    "coef-mean-rounding": ("  t = t + 0.5f;", "  t = t - 0.5f;"),
    "coef-skip-rule": ("if (!(b >= 0.05f)) { bins[c] = 0xFF; continue; }",
                       "if (!(b > 0.05f)) { bins[c] = 0xFF; continue; }"),
    "calib-scale": ("uint64_t q = nc ? (S << 16) / nc : 0;", "uint64_t q = nc ? (S << 15) / nc : 0;"),
    "calib-skips-token-0": ("      for (uint64_t t = 0; t < nc; t++) {\n        uint64_t idx = (s * T + t) * D + d;",
                            "      for (uint64_t t = 1; t < nc; t++) {\n        uint64_t idx = (s * T + t) * D + d;"),
    "renorm-threshold": ("uint64_t x_max = (((uint64_t)RANS_L >> prob_bits) << 16) * fr;",
                         "uint64_t x_max = (((uint64_t)RANS_L >> prob_bits) << 15) * fr;"),
    "state-word-order": ("  out[0] = (uint16_t)(e->x >> 16);\n  out[1] = (uint16_t)(e->x & 0xFFFF);",
                         "  out[0] = (uint16_t)(e->x & 0xFFFF);\n  out[1] = (uint16_t)(e->x >> 16);"),
    "pushed-words-forward": ("for (uint64_t k = 0; k < e->n; k++) out[2 + k] = e->buf[e->n - 1 - k];",
                             "for (uint64_t k = 0; k < e->n; k++) out[2 + k] = e->buf[k];"),
    "lanes-single-positions": ("uint64_t G = or_group(p), n = 0;", "uint64_t G = 1, n = 0;"),
    "lanes-groups-of-32-bytes": ("uint64_t G = or_group(p), n = 0;", "uint64_t G = 2 * or_group(p), n = 0;"),
    "lane-offsets-words": ("      off += 2ull * lw[l];\n    }\n  }\n  lane_offsets[nch * LANES] = off;",
                           "      off += 2ull * lw[l];\n    }\n  }\n  lane_offsets[nch * LANES] = off / 2;"),
    "model1-exponent-bits": ("o->table = p->model == 1u ? or_model1_table(bins[c], (pb >> 3) & 15u) : bins[c];",
                             "o->table = p->model == 1u ? or_model1_table(bins[c], (pb >> 4) & 15u) : bins[c];"),
    "ctx-clamp": ("x[c] = clamp64(a + b, -127, 127);", "x[c] = clamp64(a - b, -127, 127);"),
}


def run_one(name, tmp):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    if src.count(old) != 1:
        return "BAD-PATTERN", ""
    cpath = os.path.join(tmp, f"{name}.c")
    lpath = os.path.join(tmp, f"lib_{name}.so")
    open(cpath, "w").write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-w", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", lpath, cpath, "-lm"])
    env = dict(os.environ, SKV_ORACLE_LIB=lpath)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu and not slow",
                        "-p", "no:cacheprovider", *PIN_TESTS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode == 0:
        return "SURVIVED", ""
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED") or ln.startswith("ERROR")]
    return "caught", failed[0][:110] if failed else r.stdout.strip().splitlines()[-1][:110]


def main(argv):
    names = argv[1:] or list(MUTATIONS)
    survived = 0
    with tempfile.TemporaryDirectory() as tmp:
        for name in names:
            verdict, detail = run_one(name, tmp)
            survived += verdict != "caught"
            print(f"{name:28s} {verdict:11s} {detail}", flush=True)
    print(f"{len(names) - survived}/{len(names)} mutations caught")
    return 1 if survived else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
