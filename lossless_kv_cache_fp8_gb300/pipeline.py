"""Coding a KV cache held in host memory, with the host transfers overlapped.

A thin holder for the library's host-resident calls (``skv_encode_host`` /
``skv_decode_host`` in include/skv.h): the cache is coded in layer groups on
three CUDA streams (copy in, code, copy out) inside libskv.so, and the stream
and lane offsets come back byte-identical to one whole-cache call.  This class
only owns the device buffers (workspace, tables, bins) and the streams, which
the calls take from the caller; every step runs in the library.
"""
from __future__ import annotations

from . import native


class HostPipeline:
    """Round trips of one KV cache shape whose target and prediction live in pinned
    host memory.  ``group_layers`` layers are in flight per stage; the device
    holds two groups of inputs and streams, one encode workspace, the tables and
    the bins.  A group's stream buffer holds its worst case, or ``cap_frac`` of
    its raw bytes (a group that needs more fails with SKV_ERR_CAPACITY)."""

    def __init__(self, params, group_layers: int = 8, device="cuda", cap_frac: float | None = None):
        import torch
        if params.dtype not in (native.SKV_FP8_E4M3, native.SKV_BF16):
            raise ValueError("HostPipeline codes KV caches (FP8 or BF16)")
        native._check(native.skv_check_params(params), "skv_check_params")
        self.torch = torch
        self.p = params
        self.dev = torch.device(device)
        L = params.n_layers
        self.group_layers = g = max(1, min(group_layers, L))
        self.groups = [(lo, min(lo + g, L)) for lo in range(0, L, g)]
        esz = 1 if params.dtype == native.SKV_FP8_E4M3 else 2
        group_raw = g * params.n_kv * params.n_heads * params.n_tokens * params.head_dim * esz
        self.group_cap = 0 if cap_frac is None else max(4096, int(group_raw * cap_frac))
        ws = native.skv_host_workspace_bytes(params, g, self.group_cap)
        if ws == 0:
            raise ValueError("unsupported parameters for the host pipeline")
        full = native.sizes(params)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.dev)
        self.tables = torch.empty(full["tables_bytes"], dtype=torch.uint8, device=self.dev)
        self.bins = torch.empty(max(full["channels"], 16), dtype=torch.uint8, device=self.dev)
        self.streams = [torch.cuda.Stream(self.dev) for _ in range(3)]   # copy in, code, copy out
        self.n_lanes = full["lanes"]
        self.status = native.SKV_OK

    def encode(self, h_target, h_pred, h_bitstream, h_offsets, cap_bytes: int | None = None) -> int:
        """calibrate + encode the host cache; whole-cache offsets land in
        h_offsets (n_lanes + 1, int64 view of u64).  Returns the stream size."""
        torch = self.torch
        code = self.streams[1]
        code.wait_stream(torch.cuda.current_stream(self.dev))
        native._check(native.skv_build_tables(self.p, self.tables, stream=code), "skv_build_tables")
        cap = h_bitstream.numel() if cap_bytes is None else cap_bytes
        st, total = native.skv_encode_host(self.p, h_target, h_pred, self.tables, self.bins, h_bitstream, cap,
                                           h_offsets, self.group_layers, self.group_cap, self.workspace,
                                           self.streams)
        self.status = st
        native._check(st, "skv_encode_host")
        return total

    def decode(self, h_bitstream, n_bytes: int, h_offsets, h_pred, h_target_out) -> None:
        """decode the host stream against the host prediction into h_target_out
        (tables and bins from the last encode)"""
        st = native.skv_decode_host(self.p, h_bitstream, n_bytes, h_offsets, h_pred, self.tables, self.bins,
                                    h_target_out, self.group_layers, self.group_cap, self.workspace, self.streams)
        self.status = st
        native._check(st, "skv_decode_host")

    def run(self, h_target, h_pred, h_bitstream, h_offsets, decode_into=None) -> int:
        """encode, then (when `decode_into`, a host tensor, is given) decode back
        into it.  Returns the stream's byte count."""
        n = self.encode(h_target, h_pred, h_bitstream, h_offsets)
        if decode_into is not None:
            self.decode(h_bitstream, n, h_offsets, h_pred, decode_into)
        return n

    def check(self) -> int:
        """status of the last call (the host calls are synchronous)"""
        return self.status


_HOST_BUFFERS = []   # (address, bytes) of the registered mappings (kept until the process exits)


def pinned_empty(shape, dtype):
    """A host tensor in page-locked memory backed by transparent huge pages where
    the kernel offers them (an anonymous mapping advised MADV_HUGEPAGE, touched,
    then registered with cudaHostRegister), for caches of tens of GB that cross
    the host link (huge pages: far fewer page mappings behind each copy).
    Falls back to torch's pinned allocation if the mapping or the
    registration fails.  The memory lives until the process exits."""
    import ctypes
    import ctypes.util
    import mmap

    import numpy as np
    import torch

    n = 1
    for s in shape:
        n *= int(s)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    size = (nbytes + (2 << 20) - 1) & ~((2 << 20) - 1)
    libc = ctypes.CDLL(ctypes.util.find_library("c"), use_errno=True)
    libc.mmap.restype = ctypes.c_void_p
    libc.mmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long]
    libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    libc.munmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    addr = libc.mmap(None, size, mmap.PROT_READ | mmap.PROT_WRITE, mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS, -1, 0)
    if addr in (None, ctypes.c_void_p(-1).value):
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    libc.madvise(addr, size, 14)   # MADV_HUGEPAGE; advisory, ignored where unsupported
    raw = np.ctypeslib.as_array((ctypes.c_uint8 * size).from_address(addr))
    raw[:] = 0                     # fault every page in before registering
    cudart = torch.cuda.cudart()
    if cudart.cudaHostRegister(addr, size, 0) != cudart.cudaError.success:
        libc.munmap(addr, size)
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    _HOST_BUFFERS.append((addr, size))
    return torch.from_numpy(raw[:nbytes]).view(dtype).view(shape)

