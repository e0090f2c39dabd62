"""Coding a KV cache held in host memory, with the host transfers overlapped.

A range of layers is an independent sub-cache: chunks never straddle a
(layer, kv, head) slice, calibration is per channel and the tables depend only
on the dtype.  So the cache is coded in layer groups on three CUDA streams:
while group k is calibrated, encoded (and, for a round trip, decoded) on the
compute stream, group k + 1 is copied to the GPU and group k - 1's stream is
copied back.  Group streams are laid end to end in the host buffer, which is
then byte-identical to one whole-cache call (``shard.join_offsets`` rebases
the per-group lane offsets into the whole-cache offsets).

Every coding step is a call into libskv.so (``native``); torch provides the
device buffers, pinned host memory, streams and events.
"""
from __future__ import annotations

import numpy as np

from . import native, shard


class HostPipeline:
    """Round trips of one KV cache shape whose target and prediction live in pinned
    host memory.  ``group_layers`` layers are in flight per stage; device memory
    holds two groups of inputs and streams, one workspace and the tables.  A
    group's stream buffer holds its worst case, or ``cap_frac`` of its raw bytes
    (a group that needs more fails with SKV_ERR_CAPACITY)."""

    def __init__(self, params, group_layers: int = 8, device="cuda", cap_frac: float | None = None):
        import torch
        if params.dtype not in (native.SKV_FP8_E4M3, native.SKV_BF16):
            raise ValueError("HostPipeline codes KV caches (FP8 or BF16)")
        native._check(native.skv_check_params(params), "skv_check_params")
        self.torch = torch
        self.p = params
        self.dev = torch.device(device)
        L = params.n_layers
        g = max(1, min(group_layers, L))
        self.groups = [(lo, min(lo + g, L)) for lo in range(0, L, g)]
        self.gparams = [shard.shard_params(params, lo, hi) for lo, hi in self.groups]
        self.gsizes = [native.sizes(q) for q in self.gparams]
        esz = 1 if params.dtype == native.SKV_FP8_E4M3 else 2
        self.esz = esz
        self.tdt = torch.uint8 if esz == 1 else torch.int16
        self.layer_elems = params.n_kv * params.n_heads * params.n_tokens * params.head_dim
        max_elems = max(hi - lo for lo, hi in self.groups) * self.layer_elems
        # stream buffer per group: the worst case unless a fraction of the raw bytes is given
        worst = max(s["max_bitstream"] for s in self.gsizes)
        cap = worst if cap_frac is None else int(max_elems * esz * cap_frac)
        cap = max(16, (cap + 15) // 16 * 16)
        self.cap = cap
        dev = self.dev
        self.t_dev = [torch.empty(max_elems, dtype=self.tdt, device=dev) for _ in range(2)]
        self.p_dev = [torch.empty(max_elems, dtype=self.tdt, device=dev) for _ in range(2)]
        self.bs_dev = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(2)]
        max_lanes = max(s["lanes"] for s in self.gsizes)
        self.off_dev = [torch.empty(max_lanes + 1, dtype=torch.int64, device=dev) for _ in range(2)]
        full = native.sizes(params)
        self.tables = torch.empty(full["tables_bytes"], dtype=torch.uint8, device=dev)
        self.bins = torch.empty(max(full["channels"], 16), dtype=torch.uint8, device=dev)
        self.workspace = torch.empty(max(max(s["workspace"] for s in self.gsizes), 256), dtype=torch.uint8,
                                     device=dev)
        # status words per group and call (each encode / decode call clears its own)
        self.status = torch.zeros((len(self.groups), 2, 4), dtype=torch.int32, device=dev)
        self.s_in = torch.cuda.Stream(dev)
        self.s_comp = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        self.n_lanes = full["lanes"]
        self.bases = None
        self.group_bytes = None

    def _slice(self, h, k):
        lo, hi = self.groups[k]
        return h.view(-1)[lo * self.layer_elems:hi * self.layer_elems]

    def run(self, h_target, h_pred, h_bitstream, h_offsets, decode_into=None, stream=None) -> int:
        """Calibrate, build tables, encode (and decode into the device tensor
        `decode_into` when given) the cache in `h_target` / `h_pred` (pinned host
        tensors, layer-major), writing the joined stream into `h_bitstream` and
        each group's lane offsets, relative to that group's stream, into
        `h_offsets` (``self.bases`` holds the groups' byte offsets; see
        ``joined_offsets``).  `stream` (default: torch's current stream) waits
        for the whole round trip.  Returns the stream's byte count."""
        torch = self.torch
        G = len(self.groups)
        ev_in = [torch.cuda.Event() for _ in range(G)]
        ev_enc = [torch.cuda.Event() for _ in range(G)]
        ev_comp = [torch.cuda.Event() for _ in range(G)]
        ev_out = [torch.cuda.Event() for _ in range(G)]
        caller = torch.cuda.current_stream(self.dev) if stream is None else stream
        start = torch.cuda.Event()
        start.record(caller)
        for s in (self.s_in, self.s_comp, self.s_out):
            s.wait_event(start)
        h_off = h_offsets.view(-1)

        def h2d(k):
            b = k % 2
            n = (self.groups[k][1] - self.groups[k][0]) * self.layer_elems
            with torch.cuda.stream(self.s_in):
                if k >= 2:
                    self.s_in.wait_event(ev_comp[k - 2])   # buffers b were last read by group k - 2
                self.t_dev[b][:n].copy_(self._slice(h_target, k), non_blocking=True)
                self.p_dev[b][:n].copy_(self._slice(h_pred, k), non_blocking=True)
                ev_in[k].record(self.s_in)

        native._check(native.skv_build_tables(self.p, self.tables, stream=self.s_comp), "skv_build_tables")
        h2d(0)
        base, lane0 = 0, 0
        bases, sizes = [], []
        for k in range(G):
            if k + 1 < G:
                h2d(k + 1)
            b = k % 2
            q = self.gparams[k]
            lanes = self.gsizes[k]["lanes"]
            n = (self.groups[k][1] - self.groups[k][0]) * self.layer_elems
            t, p = self.t_dev[b][:n], self.p_dev[b][:n]
            sc = self.s_comp
            sc.wait_event(ev_in[k])
            if k >= 2:
                sc.wait_event(ev_out[k - 2])                 # stream buffer b copied out
            native._check(native.skv_calibrate(q, t, p, self.bins, stream=sc), "skv_calibrate")
            st, total = native.skv_encode(q, t, p, self.tables, self.bins, self.bs_dev[b], self.cap,
                                          self.off_dev[b], self.workspace, self.workspace.numel(),
                                          self.status[k, 0], want_total=True, stream=sc)
            native._check(st, "skv_encode")
            ev_enc[k].record(sc)
            if decode_into is not None:
                out = decode_into.view(-1)[self.groups[k][0] * self.layer_elems:self.groups[k][1] * self.layer_elems]
                native._check(native.skv_decode(q, self.bs_dev[b], total, self.off_dev[b], p, self.tables,
                                                self.bins, out, self.status[k, 1], stream=sc), "skv_decode")
            ev_comp[k].record(sc)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_enc[k])
                h_bitstream[base:base + total].copy_(self.bs_dev[b][:total], non_blocking=True)
                h_off[lane0:lane0 + lanes + 1].copy_(self.off_dev[b][:lanes + 1], non_blocking=True)
                ev_out[k].record(self.s_out)
            bases.append(base)
            sizes.append(total)
            base += total
            lane0 += lanes
        for e in (ev_out[G - 1], ev_comp[G - 1]):
            caller.wait_event(e)
        self.bases = bases
        self.group_bytes = sizes
        return base

    def check(self, stream=None) -> int:
        """first non-OK status of the groups of the last round trip (SKV_OK if none)"""
        for k in range(len(self.groups)):
            for c in range(2):
                st = native.skv_read_status(self.status[k, c], stream)
                if st != native.SKV_OK:
                    return st
        return native.SKV_OK

    def joined_offsets(self, h_offsets) -> np.ndarray:
        """whole-cache lane offsets (n_lanes + 1) from the per-group offsets that
        `run` wrote (host side, after the round trip has completed)"""
        h = np.asarray(h_offsets).reshape(-1).view(np.uint64)
        parts, lane0 = [], 0
        for k, (n_bytes, s) in enumerate(zip(self.group_bytes, self.gsizes)):
            lanes = s["lanes"]
            parts.append(shard.Shard(h[lane0:lane0 + lanes + 1].copy(), n_bytes))
            lane0 += lanes
        return shard.join_offsets(parts)
