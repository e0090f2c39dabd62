"""Host checks of the integer identity the CUDA encoder step rests on, and of
the table-layout constants the Python binding mirrors from include/skv.h.

The encoder entry of a symbol with frequency fr holds m = 2^32 + m_lo =
ceil(2^(32+s) / fr) with s = ceil(log2 fr), which puts m in [2^32, 2^33),
and the kernel evaluates floor(x / fr) as (umulhi(x, m_lo) + x) >> s for
every state x below the renormalisation threshold fr * 2^20.  The exact
condition is checked directly at the states that decide it (x = k fr - 1,
the largest state below each multiple, up to k = 2^20), plus random states,
for every frequency 1..4095.
"""
import random
import re

from lossless_kv_cache_fp8_gb300 import native


def _entry(fr):
    s = (fr - 1).bit_length()           # ceil(log2 fr)
    k = 1 << (32 + s)
    m = -(-k // fr)
    assert (1 << 32) <= m < (1 << 33), fr
    x1 = fr * (1 << 20) - 1
    assert x1 * (m * fr - k) < k and x1 * m < (1 << 64), fr
    return m, s


def _kernel_quot(x, m, s):
    m_lo = m & 0xFFFFFFFF
    t = ((x * m_lo) >> 32) + x
    assert t < (1 << 32)            # the kernel adds in 32 bits
    return t >> s


def test_reciprocal_matches_division_below_threshold():
    rng = random.Random(7)
    for fr in range(1, 4096):
        m, s = _entry(fr)
        e = m * fr - (1 << (32 + s))
        # floor((k fr - 1) m / 2^(32+s)) = k - 1 for all k <= 2^20  <=>  2^20 e < m
        assert (1 << 20) * e < m, fr
        for x in [fr * (1 << 20) - 1, (1 << 16), fr * 7 - 1, fr * 7] + [rng.randrange(1 << 16, fr << 20) for _ in range(6)]:
            if (1 << 16) <= x < fr << 20:
                assert _kernel_quot(x, m, s) == x // fr, (fr, x)


def test_coded_state_stays_in_range():
    # after renormalisation x < fr 2^20, so x' = (x // fr) 4096 + x % fr + cum < 2^32
    for fr in range(1, 4096):
        x = fr * (1 << 20) - 1
        cum = 4096 - fr
        assert (x // fr) * 4096 + x % fr + cum < (1 << 32)
        x = (1 << 16)
        assert (x // fr) * 4096 + x % fr >= (1 << 16)


def _header_defines():
    txt = open(native.HEADER).read()
    return {k: int(v, 0) for k, v in re.findall(r"#define\s+(SKV_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", txt)}


def test_binding_constants_match_header():
    h = _header_defines()
    names = ["SKV_TABLE_STRIDE", "SKV_TABLE_SLOT_BYTES", "SKV_TABLE_ENC_OFF", "SKV_TABLE_LUT_OFF", "SKV_TABLE_DEC_OFF",
             "SKV_TABLE_FREQ_OFF", "SKV_TABLE_CUM_OFF", "SKV_OK", "SKV_ERR_INVALID_ARG", "SKV_ERR_CUDA",
             "SKV_ERR_CAPACITY", "SKV_ERR_CORRUPT", "SKV_ERR_TIMEOUT", "SKV_ERR_UNSUPPORTED",
             "SKV_FP8_E4M3", "SKV_BF16", "SKV_COEF_I16"]
    for n in names:
        assert getattr(native, n) == h[n], n
    # regions are 16-byte aligned, disjoint and inside the stride
    regions = sorted([(h["SKV_TABLE_ENC_OFF"], 2048), (h["SKV_TABLE_LUT_OFF"], 4096), (h["SKV_TABLE_DEC_OFF"], 1024),
                      (h["SKV_TABLE_FREQ_OFF"], 512), (h["SKV_TABLE_CUM_OFF"], 514)])
    for (o1, n1), (o2, _) in zip(regions, regions[1:]):
        assert o1 % 16 == 0 and o1 + n1 <= o2
    assert regions[-1][0] + regions[-1][1] <= h["SKV_TABLE_STRIDE"] and h["SKV_TABLE_STRIDE"] % 16 == 0
