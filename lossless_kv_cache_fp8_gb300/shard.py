"""Splitting one KV cache across ranks by layers and joining the shard streams.

Chunks never straddle a (layer, kv, head) slice and calibration is per channel,
so a layer range is an independent sub-cache: each rank calibrates, builds the
same tables and codes its layers with no exchange of data.  The only collective
is an all-gather of the per-shard byte totals, which places each shard's stream
in the joined stream and rebases its lane offsets; the joined stream is then
byte-identical to coding the whole cache on one GPU.
"""
from __future__ import annotations

import dataclasses

import numpy as np


def layer_ranges(n_layers: int, world: int):
    """contiguous layer range [lo, hi) of every rank (the first ranks take one more)"""
    base, extra = divmod(n_layers, world)
    out, lo = [], 0
    for r in range(world):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def shard_params(params, lo: int, hi: int):
    """skv_params (or the oracle's params) of layers [lo, hi)"""
    q = type(params).from_buffer_copy(params)
    q.n_layers = hi - lo
    return q


@dataclasses.dataclass
class Shard:
    lane_offsets: np.ndarray   # uint64, n_lanes + 1, relative to the shard's stream
    n_bytes: int


def shard_bases(totals):
    """byte offset of every shard's stream in the joined stream"""
    return np.concatenate([[0], np.cumsum(np.asarray(totals, dtype=np.uint64))[:-1]]).astype(np.uint64)


def join_offsets(shards):
    """lane offsets of the joined stream from the shards' own offsets"""
    bases = shard_bases([s.n_bytes for s in shards])
    parts = [s.lane_offsets[:-1].astype(np.uint64) + b for s, b in zip(shards, bases)]
    total = int(sum(s.n_bytes for s in shards))
    return np.concatenate(parts + [np.array([total], dtype=np.uint64)])


def gather_totals(local_total: int, group=None):
    """all-gather of the per-shard byte totals (the one collective)"""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([local_total], dtype=torch.int64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t, group=group)
    return [int(x.item()) for x in out]


def encode_layer_shard(params, target, pred, lo: int, hi: int, group=None, device=None, cap_frac: float = 1.0):
    """One rank's part of a sharded encode through the CUDA library: calibrate,
    build the tables and encode layers [lo, hi) (``target`` / ``pred`` hold only
    those layers, on this rank's GPU), then all-gather the byte totals.

    Returns (codec, n_bytes, base, totals): the shard's stream is
    ``codec.bitstream[:n_bytes]`` and belongs at byte ``base`` of the joined
    stream; its lane offsets plus ``base`` are the joined offsets of its lanes
    (lanes are numbered layer-major, so shard r's lanes follow shard r-1's)."""
    from . import native
    q = shard_params(params, lo, hi)
    raw = target.numel() * target.element_size()
    cap = None if cap_frac >= 1.0 else max(4096, int(raw * cap_frac))
    codec = native.Codec(q, device=device or target.device, bitstream_capacity=cap)
    codec.calibrate(target, pred)
    codec.build_tables()
    n = codec.encode(target, pred, want_total=True)
    native._check(codec.check(), "skv_encode (shard)")
    totals = gather_totals(n, group)
    import torch.distributed as dist
    rank = dist.get_rank(group)
    return codec, n, int(shard_bases(totals)[rank]), totals
