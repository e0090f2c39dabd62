"""CPU oracle for speculative KV coding -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The oracle itself is plain single-threaded C (``skv_oracle.c``), compiled here
with gcc; this module only marshals numpy arrays into it.  Each C function
cites the page passage it follows.  Pins that fix it independently of its own
code live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "skv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libskv_oracle.so")

FP8, BF16, COEF = 1, 2, 3
OK, ERR_ARG, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 3, 4
LANES = 32


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Params(C.Structure):
    _fields_ = [("version", C.c_uint32), ("dtype", C.c_uint32), ("n_layers", C.c_uint32),
                ("n_kv", C.c_uint32), ("n_heads", C.c_uint32), ("head_dim", C.c_uint32),
                ("n_tokens", C.c_uint64), ("n_coef", C.c_uint32), ("lane_syms", C.c_uint32),
                ("n_calib", C.c_uint32), ("model", C.c_uint32)]


def kv_params(dtype: int, n_layers: int, n_kv: int, n_heads: int, head_dim: int,
              n_tokens: int, lane_syms: int, n_calib: int = 256, model: int = 0) -> Params:
    return Params(1, dtype, n_layers, n_kv, n_heads, head_dim, n_tokens, 0, lane_syms, n_calib, model)


def coef_params(n_tokens: int, n_coef: int, lane_syms: int) -> Params:
    return Params(1, COEF, 0, 0, 0, 0, n_tokens, n_coef, lane_syms, 0, 0)


_lib = None


def lib():
    global _lib
    if _lib is None:
        # SKV_ORACLE_LIB: a different build of the same source (the mutation
        # check of tests/oracle_mutations.py loads copies with planted mistakes)
        _lib = C.CDLL(os.environ.get("SKV_ORACLE_LIB") or build())
        P = C.POINTER(Params)
        vp = C.c_void_p
        u64, u32, i32 = C.c_uint64, C.c_uint32, C.c_int
        sig = {
            "or_ordinal": (u32, [u32, u32]), "or_ordinal_inv": (u32, [u32, u32]),
            "or_bin_from_q": (u32, [u64, u32]), "or_beta_q": (u64, [u32, u32]),
            "or_bin_ext": (u32, [u64]), "or_model1_table": (u32, [u32, u32]),
            "or_ctx_means": (i32, [u32, u32, vp, vp, u32, u32, vp, u64, vp, u64, vp]),
            "or_tau_q": (u64, [u64]), "or_power_chain": (None, [u64, vp]),
            "or_masses": (None, [u32, u32, u32, vp]),
            "or_build_table": (None, [u32, u32, u32, vp, vp]),
            "or_build_tables": (i32, [P, vp, vp]),
            "or_num_tables": (u32, [P]), "or_sub_bins": (u32, [P]), "or_group": (u32, [P]),
            "or_num_slices": (u64, [P]), "or_slice_positions": (u64, [P]),
            "or_chunks_per_slice": (u64, [P]), "or_num_chunks": (u64, [P]),
            "or_num_lanes": (u64, [P]), "or_num_channels": (u64, [P]),
            "or_max_lane_words": (u64, [P]), "or_check_params": (i32, [P]),
            "or_calibrate": (i32, [P, vp, vp, vp, vp, vp]),
            "or_rans_encode": (i32, [u32, vp, vp, vp, u64, vp, u64, vp]),
            "or_rans_decode": (i32, [u32, vp, vp, u32, vp, u64, u64, vp]),
            "or_encode_chunk": (i32, [P, u64, vp, vp, vp, vp, vp, vp, u64, vp]),
            "or_decode_chunk": (i32, [P, u64, vp, vp, vp, vp, vp, vp, vp]),
            "or_encode": (i32, [P, vp, vp, vp, vp, vp, vp, u64, vp, vp]),
            "or_decode": (i32, [P, vp, vp, vp, vp, u64, vp, vp, vp]),
            "or_shannon_bits": (C.c_double, [P, vp, vp, vp, vp]),
            "or_symbols": (i32, [P, vp, vp, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- scalar maps ---------------------------------------------------------------------------
def ordinal(bits: int, width: int) -> int:
    return lib().or_ordinal(bits, width)


def ordinal_inv(u: int, width: int) -> int:
    return lib().or_ordinal_inv(u, width)


def bin_from_q(q: int, sub: int) -> int:
    return lib().or_bin_from_q(q, sub)


def beta_q(b: int, sub: int) -> int:
    return lib().or_beta_q(b, sub)


def tau_q(bq: int) -> int:
    return lib().or_tau_q(bq)


def power_chain(tq: int) -> np.ndarray:
    P = np.zeros(2056, np.uint64)
    lib().or_power_chain(tq, _ptr(P))
    return P


def masses(b: int, sub: int, f: int) -> np.ndarray:
    m = np.zeros(256, np.uint64)
    lib().or_masses(b, sub, f, _ptr(m))
    return m


def build_table(b: int, sub: int, f: int):
    fr = np.zeros(256, np.uint16)
    cum = np.zeros(257, np.uint16)
    lib().or_build_table(b, sub, f, _ptr(fr), _ptr(cum))
    return fr, cum


# --- geometry ------------------------------------------------------------------------------
def geometry(p: Params) -> dict:
    L = lib()
    return dict(n_tables=L.or_num_tables(C.byref(p)), sub=L.or_sub_bins(C.byref(p)),
                group=L.or_group(C.byref(p)), n_slices=L.or_num_slices(C.byref(p)),
                slice_positions=L.or_slice_positions(C.byref(p)),
                chunks_per_slice=L.or_chunks_per_slice(C.byref(p)),
                n_chunks=L.or_num_chunks(C.byref(p)), n_lanes=L.or_num_lanes(C.byref(p)),
                n_channels=L.or_num_channels(C.byref(p)),
                max_lane_words=L.or_max_lane_words(C.byref(p)))


def check_params(p: Params) -> int:
    return lib().or_check_params(C.byref(p))


# --- pipeline ------------------------------------------------------------------------------
def calibrate(p: Params, target, pred, want_sum=True, want_hist=False):
    """KV: target/pred raw-bit arrays (uint8 or uint16).  COEF: target=None,
    pred=beta_c fp32.  Returns (bins, sum_abs or None, hist or None)."""
    g = geometry(p)
    nch = g["n_channels"]
    bins = np.zeros(nch, np.uint8)
    s = np.zeros(nch, np.uint32) if (want_sum and p.dtype != COEF) else None
    h = np.zeros((nch, 256), np.uint32) if (want_hist and p.dtype != COEF) else None
    st = lib().or_calibrate(C.byref(p), _ptr(target), _ptr(pred), _ptr(bins), _ptr(s), _ptr(h))
    if st != OK:
        raise ValueError(f"or_calibrate status {st}")
    return bins, s, h


def build_tables(p: Params):
    nt = geometry(p)["n_tables"]
    fr = np.zeros((nt, 256), np.uint16)
    cum = np.zeros((nt, 257), np.uint16)
    st = lib().or_build_tables(C.byref(p), _ptr(fr), _ptr(cum))
    if st != OK:
        raise ValueError(f"or_build_tables status {st}")
    return fr, cum


def max_bitstream_bytes(p: Params) -> int:
    g = geometry(p)
    return 2 * g["n_lanes"] * g["max_lane_words"]


def encode(p: Params, freq, cum, bins, target, pred, cap_bytes: int | None = None):
    """Returns (bitstream uint8[total], lane_offsets uint64[n_lanes+1])."""
    g = geometry(p)
    cap = max_bitstream_bytes(p) if cap_bytes is None else cap_bytes
    bs = np.zeros(cap + 2, np.uint8)
    offs = np.zeros(g["n_lanes"] + 1, np.uint64)
    tot = np.zeros(1, np.uint64)
    st = lib().or_encode(C.byref(p), _ptr(freq), _ptr(cum), _ptr(bins), _ptr(target), _ptr(pred),
                         _ptr(bs), cap, _ptr(offs), _ptr(tot))
    if st != OK:
        return st, None, None
    return OK, bs[: int(tot[0])].copy(), offs


def decode(p: Params, freq, cum, bins, bitstream, lane_offsets, pred, out_dtype):
    n_pos = geometry(p)["n_slices"] * geometry(p)["slice_positions"]
    out = np.zeros(n_pos, out_dtype)
    bs = np.ascontiguousarray(bitstream)
    if bs.size == 0:
        bs = np.zeros(2, np.uint8)
    st = lib().or_decode(C.byref(p), _ptr(freq), _ptr(cum), _ptr(bins), _ptr(bs),
                         int(np.asarray(bitstream).size), _ptr(_c(lane_offsets, np.uint64)),
                         _ptr(pred), _ptr(out))
    return st, out


def encode_chunk(p: Params, chunk: int, freq, cum, bins, tgt_chunk, pred_chunk):
    """Encode one chunk from its own data (chunk-relative arrays).
    Returns (words uint16[...], lane_words uint32[32])."""
    cap = LANES * geometry(p)["max_lane_words"]
    out = np.zeros(cap, np.uint16)
    lw = np.zeros(LANES, np.uint32)
    st = lib().or_encode_chunk(C.byref(p), chunk, _ptr(freq), _ptr(cum), _ptr(bins),
                               _ptr(tgt_chunk), _ptr(pred_chunk), _ptr(out), cap, _ptr(lw))
    if st != OK:
        raise ValueError(f"or_encode_chunk status {st}")
    return out[: int(lw.sum())].copy(), lw


def decode_chunk(p: Params, chunk: int, freq, cum, bins, words, lane_words, pred_chunk, n_pos, out_dtype):
    out = np.zeros(n_pos, out_dtype)
    w = np.ascontiguousarray(words, np.uint16)
    if w.size == 0:
        w = np.zeros(1, np.uint16)
    st = lib().or_decode_chunk(C.byref(p), chunk, _ptr(freq), _ptr(cum), _ptr(bins), _ptr(w),
                               _ptr(_c(lane_words, np.uint32)), _ptr(pred_chunk), _ptr(out))
    return st, out


def shannon_bits(p: Params, freq, bins, target, pred) -> float:
    return lib().or_shannon_bits(C.byref(p), _ptr(freq), _ptr(bins), _ptr(target), _ptr(pred))


def symbols(p: Params, bins, target, pred):
    g = geometry(p)
    n = g["n_slices"] * g["slice_positions"]
    t = np.zeros(n, np.uint32)
    s = np.zeros(n, np.int32)
    r = np.zeros(n, np.uint32)
    st = lib().or_symbols(C.byref(p), _ptr(bins), _ptr(target), _ptr(pred), _ptr(t), _ptr(s), _ptr(r))
    if st != OK:
        raise ValueError(f"or_symbols status {st}")
    return t, s, r


# --- generic coder over an arbitrary table (hand examples, brute force) --------------------
def rans_encode(prob_bits: int, freq, cum, syms):
    f = _c(freq, np.uint32)
    c = _c(cum, np.uint32)
    s = _c(syms, np.uint32)
    cap = 2 * len(s) + 4
    out = np.zeros(cap, np.uint16)
    n = np.zeros(1, np.uint64)
    st = lib().or_rans_encode(prob_bits, _ptr(f), _ptr(c), _ptr(s) if len(s) else None, len(s),
                              _ptr(out), cap, _ptr(n))
    if st != OK:
        raise ValueError(f"or_rans_encode status {st}")
    return out[: int(n[0])].copy()


def rans_decode(prob_bits: int, freq, cum, words, n: int):
    f = _c(freq, np.uint32)
    c = _c(cum, np.uint32)
    w = _c(words, np.uint16)
    out = np.zeros(max(n, 1), np.uint32)
    st = lib().or_rans_decode(prob_bits, _ptr(f), _ptr(c), len(f), _ptr(w), len(w), n, _ptr(out))
    return st, out[:n]


def ctx_means(V, U, s1, s2, q_even, mu_odd):
    """odd rows' context-shifted means (float32 [n_odd][C]) from the even rows"""
    V = np.ascontiguousarray(V, np.int8)
    U = np.ascontiguousarray(U, np.int8)
    qe = np.ascontiguousarray(q_even, np.int16)
    mo = np.ascontiguousarray(mu_odd, np.float32)
    R, C = V.shape
    out = np.zeros(mo.shape, np.float32)
    st = lib().or_ctx_means(C, R, _ptr(V), _ptr(U), s1, s2, _ptr(qe), qe.shape[0], _ptr(mo), mo.shape[0],
                            _ptr(out))
    if st != OK:
        raise ValueError(f"or_ctx_means status {st}")
    return out
