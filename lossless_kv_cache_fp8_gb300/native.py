"""Thin ctypes binding of libskv.so (the C ABI declared in include/skv.h).

Functions keep the C names and only marshal arguments: tensors become device
pointers (``data_ptr()``), ``stream=None`` becomes torch's current CUDA stream.
Every step of the coding path runs in the library's CUDA kernels; if the
library is missing this module raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes as C
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "_build", "libskv.so")
HEADER = os.path.join(ROOT, "include", "skv.h")

SKV_OK, SKV_ERR_INVALID_ARG, SKV_ERR_CUDA, SKV_ERR_CAPACITY = 0, 1, 2, 3
SKV_ERR_CORRUPT, SKV_ERR_TIMEOUT, SKV_ERR_UNSUPPORTED = 4, 5, 6
SKV_FP8_E4M3, SKV_BF16, SKV_COEF_I16 = 1, 2, 3
SKV_TABLE_STRIDE = 8704
SKV_TABLE_ENC_OFF, SKV_TABLE_LUT_OFF, SKV_TABLE_DEC_OFF = 0, 2048, 6144
SKV_TABLE_FREQ_OFF, SKV_TABLE_CUM_OFF = 7168, 7680
SKV_TABLE_SLOT_BYTES = 16384


class SkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class skv_params(C.Structure):
    _fields_ = [("version", C.c_uint32), ("dtype", C.c_uint32), ("n_layers", C.c_uint32),
                ("n_kv", C.c_uint32), ("n_heads", C.c_uint32), ("head_dim", C.c_uint32),
                ("n_tokens", C.c_uint64), ("n_coef", C.c_uint32), ("lane_syms", C.c_uint32),
                ("n_calib", C.c_uint32), ("model", C.c_uint32)]


class skv_paged_layout(C.Structure):
    _fields_ = [("d_block_table", C.c_void_p), ("n_blocks", C.c_uint32), ("block_tokens", C.c_uint32)]


class skv_ctx_map(C.Structure):
    _fields_ = [("d_V", C.c_void_p), ("d_U", C.c_void_p), ("rank", C.c_uint32), ("shift1", C.c_uint32),
                ("shift2", C.c_uint32)]


def ctx_map(V, U, shift1: int, shift2: int) -> skv_ctx_map:
    """map of int8 device tensors V [rank][n_coef], U [n_coef][rank]"""
    return skv_ctx_map(_ptr(V), _ptr(U), V.shape[0], shift1, shift2)


def paged_layout(block_table, n_blocks: int, block_tokens: int) -> skv_paged_layout:
    """layout of paged pools; block_table: a uint32-valued device tensor (int32 storage)"""
    return skv_paged_layout(_ptr(block_table), n_blocks, block_tokens)


SKV_MODEL_CHANNEL, SKV_MODEL_EXPONENT = 0, 1


def kv_params(dtype, n_layers, n_kv, n_heads, head_dim, n_tokens, lane_syms, n_calib=256, model=0) -> skv_params:
    return skv_params(1, dtype, n_layers, n_kv, n_heads, head_dim, n_tokens, 0, lane_syms, n_calib, model)


def coef_params(n_tokens, n_coef, lane_syms) -> skv_params:
    return skv_params(1, SKV_COEF_I16, 0, 0, 0, 0, n_tokens, n_coef, lane_syms, 0, 0)


def params_for(w, model: int = 0) -> skv_params:
    """skv_params of a synth.Workload"""
    if w.dtype == SKV_COEF_I16:
        return coef_params(w.n_tokens, w.n_coef, w.lane_syms)
    return kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib, model)


_lib = None
_P = C.POINTER(skv_params)
_PL = C.POINTER(skv_paged_layout)
_CM = C.POINTER(skv_ctx_map)
_SIGS = {
    "skv_status_string": (C.c_char_p, [C.c_int]),
    "skv_check_params": (C.c_int, [_P]),
    "skv_num_positions": (C.c_uint64, [_P]),
    "skv_num_channels": (C.c_uint64, [_P]),
    "skv_num_tables": (C.c_uint32, [_P]),
    "skv_num_chunks": (C.c_uint64, [_P]),
    "skv_num_lanes": (C.c_uint64, [_P]),
    "skv_tables_bytes": (C.c_uint64, [_P]),
    "skv_max_bitstream_bytes": (C.c_uint64, [_P]),
    "skv_encode_workspace_bytes": (C.c_uint64, [_P]),
    "skv_calibrate": (C.c_int, [_P, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_build_tables": (C.c_int, [_P, C.c_void_p, C.c_uint64, C.c_void_p]),
    "skv_encode": (C.c_int, [_P, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint64,
                             C.c_void_p, C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_decode": (C.c_int, [_P, C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                             C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_encode_noalloc": (C.c_int, [_P, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_selftest_ctx_wait": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_selftest_lookback": (C.c_int, [C.c_void_p, C.c_uint32, C.c_uint32, C.c_uint32, C.c_void_p, C.c_void_p,
                                        C.c_void_p]),
    "skv_read_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "skv_calibrate_paged": (C.c_int, [_P, _PL, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p]),
    "skv_encode_paged": (C.c_int, [_P, _PL, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.c_uint64, C.c_void_p, C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p,
                                   C.c_void_p]),
    "skv_decode_paged": (C.c_int, [_P, _PL, C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "skv_ctx_scratch_bytes": (C.c_uint64, [C.c_uint64, C.c_uint32, C.c_uint32]),
    "skv_host_workspace_bytes": (C.c_uint64, [_P, C.c_uint32, C.c_uint64]),
    "skv_checked_failures": (C.c_int, [C.c_void_p, C.c_void_p]),
    "skv_encode_host": (C.c_int, [_P, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint64,
                                  C.c_void_p, C.c_void_p, C.c_uint32, C.c_uint64, C.c_void_p, C.c_uint64,
                                  C.c_void_p]),
    "skv_decode_host": (C.c_int, [_P, C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_uint32, C.c_uint64, C.c_void_p, C.c_uint64, C.c_void_p]),
    "skv_ctx_means": (C.c_int, [_CM, C.c_void_p, C.c_uint64, C.c_void_p, C.c_uint64, C.c_uint32, C.c_void_p,
                                C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p]),
}


def load(path: str):
    """load a build of the library (the ordinary one, or the checked one) with
    its function signatures"""
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} not built ({path}); run __graft_entry__.build()")
    L = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """Load libskv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def use_library(path: str | None):
    """route every call of this module to another build (None: libskv.so again)"""
    global _lib
    _lib = None if path is None else load(path)


def skv_checked_failures():
    """(status, count, first site) of the checked build's failed checks (cleared)"""
    n, site = C.c_uint32(0), C.c_uint32(0)
    st = lib().skv_checked_failures(C.byref(n), C.byref(site))
    return st, n.value, site.value


def header_functions() -> list[str]:
    """names of the functions include/skv.h declares"""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(skv_[a-z_]+)\s*\(", txt)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(st: int) -> str:
    return lib().skv_status_string(st).decode()


def _check(st: int, what: str) -> int:
    if st != SKV_OK:
        raise SkvError(st, what)
    return st


# --- sizes -------------------------------------------------------------------------------------
def sizes(p: skv_params) -> dict:
    L = lib()
    r = C.byref(p)
    return dict(positions=L.skv_num_positions(r), channels=L.skv_num_channels(r),
                tables=L.skv_num_tables(r), chunks=L.skv_num_chunks(r), lanes=L.skv_num_lanes(r),
                tables_bytes=L.skv_tables_bytes(r), max_bitstream=L.skv_max_bitstream_bytes(r),
                workspace=L.skv_encode_workspace_bytes(r))


def skv_check_params(p: skv_params) -> int:
    return lib().skv_check_params(C.byref(p))


# --- the four calls (same names as the C ABI) ----------------------------------------------------
def skv_calibrate(p, target, pred, bins, sum_abs=None, hist=None, stream=None) -> int:
    return lib().skv_calibrate(C.byref(p), _ptr(target), _ptr(pred), _ptr(bins), _ptr(sum_abs),
                               _ptr(hist), _stream(stream))


def skv_build_tables(p, tables, tables_bytes=None, stream=None) -> int:
    nb = tables_bytes if tables_bytes is not None else tables.numel() * tables.element_size()
    return lib().skv_build_tables(C.byref(p), _ptr(tables), nb, _stream(stream))


def skv_encode(p, target, pred, tables, bins, bitstream, cap_bytes, lane_offsets, workspace,
               workspace_bytes, status, want_total=True, stream=None):
    """Returns (status_code, total_bytes or None)."""
    tot = C.c_uint64(0)
    st = lib().skv_encode(C.byref(p), _ptr(target), _ptr(pred), _ptr(tables), _ptr(bins), _ptr(bitstream),
                          cap_bytes, _ptr(lane_offsets), _ptr(workspace), workspace_bytes, _ptr(status),
                          C.byref(tot) if want_total else None, _stream(stream))
    return st, (tot.value if want_total else None)


def skv_encode_noalloc(p, target, pred, tables, bins, bitstream, cap_bytes, lane_offsets, status,
                       want_total=True, stream=None):
    """Encode with the library's own static scratch (no workspace argument).
    Returns (status_code, total_bytes or None)."""
    tot = C.c_uint64(0)
    st = lib().skv_encode_noalloc(C.byref(p), _ptr(target), _ptr(pred), _ptr(tables), _ptr(bins), _ptr(bitstream),
                                  cap_bytes, _ptr(lane_offsets), _ptr(status),
                                  C.byref(tot) if want_total else None, _stream(stream))
    return st, (tot.value if want_total else None)


def skv_decode(p, bitstream, n_bytes, lane_offsets, pred, tables, bins, target_out, status, stream=None) -> int:
    return lib().skv_decode(C.byref(p), _ptr(bitstream), n_bytes, _ptr(lane_offsets), _ptr(pred), _ptr(tables),
                            _ptr(bins), _ptr(target_out), _ptr(status), _stream(stream))


def skv_selftest_ctx_wait(scratch, status, stream=None) -> int:
    return lib().skv_selftest_ctx_wait(_ptr(scratch), _ptr(status), _stream(stream))


def skv_selftest_lookback(state, n_chunks, missing_chunk, max_spins, excl, status, stream=None) -> int:
    return lib().skv_selftest_lookback(_ptr(state), n_chunks, missing_chunk, max_spins, _ptr(excl), _ptr(status),
                                       _stream(stream))


def _streams3(streams):
    """array of three cudaStream_t (copy in, code, copy out) for the host calls"""
    arr = (C.c_void_p * 3)(*[_stream(s) for s in streams])
    return arr


def skv_host_workspace_bytes(p, group_layers: int, group_cap_bytes: int = 0) -> int:
    return lib().skv_host_workspace_bytes(C.byref(p), group_layers, group_cap_bytes)


def skv_encode_host(p, h_target, h_pred, tables, bins, h_bitstream, cap_bytes, h_lane_offsets, group_layers,
                    group_cap_bytes, workspace, streams):
    """returns (status, total bytes); synchronous"""
    total = C.c_uint64(0)
    st = lib().skv_encode_host(C.byref(p), _ptr(h_target), _ptr(h_pred), _ptr(tables), _ptr(bins),
                               _ptr(h_bitstream), cap_bytes, _ptr(h_lane_offsets), C.byref(total), group_layers,
                               group_cap_bytes, _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _streams3(streams))
    return st, total.value


def skv_decode_host(p, h_bitstream, n_bytes, h_lane_offsets, h_pred, tables, bins, h_target_out, group_layers,
                    group_cap_bytes, workspace, streams) -> int:
    return lib().skv_decode_host(C.byref(p), _ptr(h_bitstream), n_bytes, _ptr(h_lane_offsets), _ptr(h_pred),
                                 _ptr(tables), _ptr(bins), _ptr(h_target_out), group_layers, group_cap_bytes,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _streams3(streams))


def skv_read_status(status, stream=None) -> int:
    return lib().skv_read_status(_ptr(status), _stream(stream))


# --- checkerboard context (same names as the C ABI) ----------------------------------------------
def skv_ctx_scratch_bytes(n_odd: int, n_coef: int, rank: int) -> int:
    return lib().skv_ctx_scratch_bytes(n_odd, n_coef, rank)


def skv_ctx_means(cmap, q_even, n_even, mu_odd, n_odd, n_coef, mu_out, scratch, status, scratch_bytes=None,
                  stream=None) -> int:
    nb = scratch_bytes if scratch_bytes is not None else scratch.numel() * scratch.element_size()
    return lib().skv_ctx_means(C.byref(cmap), _ptr(q_even), n_even, _ptr(mu_odd), n_odd, n_coef, _ptr(mu_out),
                               _ptr(scratch), nb, _ptr(status), _stream(stream))


# --- paged pools (same names as the C ABI) -----------------------------------------------------
def skv_calibrate_paged(p, layout, target_pool, pred_pool, bins, status, sum_abs=None, hist=None,
                        stream=None) -> int:
    return lib().skv_calibrate_paged(C.byref(p), C.byref(layout), _ptr(target_pool), _ptr(pred_pool), _ptr(bins),
                                     _ptr(sum_abs), _ptr(hist), _ptr(status), _stream(stream))


def skv_encode_paged(p, layout, target_pool, pred_pool, tables, bins, bitstream, cap_bytes, lane_offsets,
                     workspace, workspace_bytes, status, want_total=True, stream=None):
    """Returns (status_code, total_bytes or None)."""
    tot = C.c_uint64(0)
    st = lib().skv_encode_paged(C.byref(p), C.byref(layout), _ptr(target_pool), _ptr(pred_pool), _ptr(tables),
                                _ptr(bins), _ptr(bitstream), cap_bytes, _ptr(lane_offsets), _ptr(workspace),
                                workspace_bytes, _ptr(status), C.byref(tot) if want_total else None,
                                _stream(stream))
    return st, (tot.value if want_total else None)


def skv_decode_paged(p, layout, bitstream, n_bytes, lane_offsets, pred_pool, tables, bins, target_pool_out,
                     status, stream=None) -> int:
    return lib().skv_decode_paged(C.byref(p), C.byref(layout), _ptr(bitstream), n_bytes, _ptr(lane_offsets),
                                  _ptr(pred_pool), _ptr(tables), _ptr(bins), _ptr(target_pool_out), _ptr(status),
                                  _stream(stream))


# --- convenience: device buffers from torch, the calls above, errors raised --------------------
class Codec:
    """Owns the device buffers of one stream shape; every compute step is a call
    into libskv.so.  Inputs are torch CUDA tensors of raw bits (uint8 for FP8,
    int16 for BF16 / COEF q) and fp32 for COEF means / scales."""

    def __init__(self, p: skv_params, device="cuda", bitstream_capacity: int | None = None):
        import torch
        self.p = p
        _check(skv_check_params(p), "skv_check_params")
        self.sz = sizes(p)
        self.torch = torch
        dev = torch.device(device)
        self.bins = torch.empty(max(self.sz["channels"], 16), dtype=torch.uint8, device=dev)
        self.tables = torch.empty(self.sz["tables_bytes"], dtype=torch.uint8, device=dev)
        self.lane_offsets = torch.empty(self.sz["lanes"] + 1, dtype=torch.int64, device=dev)
        self.workspace = torch.empty(max(self.sz["workspace"], 256), dtype=torch.uint8, device=dev)
        cap = self.sz["max_bitstream"] if bitstream_capacity is None else bitstream_capacity
        self.cap = int(max(cap, 16))
        self.bitstream = torch.empty(self.cap, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.n_bytes = None

    def calibrate(self, target, calib_pred, sum_abs=None, hist=None, stream=None):
        _check(skv_calibrate(self.p, target, calib_pred, self.bins, sum_abs, hist, stream), "skv_calibrate")
        return self.bins[: self.sz["channels"]]

    def build_tables(self, stream=None):
        _check(skv_build_tables(self.p, self.tables, stream=stream), "skv_build_tables")
        return self.tables

    def encode(self, target, pred, want_total=True, stream=None):
        st, tot = skv_encode(self.p, target, pred, self.tables, self.bins, self.bitstream, self.cap,
                             self.lane_offsets, self.workspace, self.workspace.numel(), self.status,
                             want_total=want_total, stream=stream)
        _check(st, "skv_encode")
        if want_total:
            self.n_bytes = tot
        return tot

    def decode(self, pred, out, bitstream=None, n_bytes=None, lane_offsets=None, stream=None):
        bs = self.bitstream if bitstream is None else bitstream
        nb = self.n_bytes if n_bytes is None else n_bytes
        lo = self.lane_offsets if lane_offsets is None else lane_offsets
        _check(skv_decode(self.p, bs, nb, lo, pred, self.tables, self.bins, out, self.status, stream),
               "skv_decode")
        return out

    def check(self, stream=None):
        return skv_read_status(self.status, stream)
