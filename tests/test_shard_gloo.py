"""Multi-rank path on CPU: two gloo ranks code layer shards of one cache (with the
oracle standing in for each rank's GPU), all-gather their byte totals and join;
the joined stream and lane offsets equal the single-process stream."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

W = dict(name="qwen3-0.6b-1k-fp8", n_layers=5, n_tokens=300, lane_syms=64)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    from lossless_kv_cache_fp8_gb300 import shard, synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.WORKLOADS[W["name"]].scaled(n_layers=W["n_layers"], n_tokens=W["n_tokens"], lane_syms=W["lane_syms"])
    lo, hi = shard.layer_ranges(w.n_layers, world)[rank]
    t, p = synth.gen_kv(w, "cpu", layers=(lo, hi))
    po = shard.shard_params(oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens,
                                             w.lane_syms, w.n_calib), lo, hi)
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    bins, _, _ = oracle.calibrate(po, tn, pn)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    totals = shard.gather_totals(int(bs.size))
    base = int(shard.shard_bases(totals)[rank])
    parts = [None] * world
    dist.all_gather_object(parts, (bs.tobytes(), offs.tolist(), base))
    if rank == 0:
        shards = [shard.Shard(np.array(o, dtype=np.uint64), len(b)) for b, o, _ in parts]
        joined = b"".join(b for b, _, _ in parts)
        q.put((joined, shard.join_offsets(shards).tolist(), [b for _, _, b in parts], totals))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_layer_shards_join_to_one_stream(orc):
    from lossless_kv_cache_fp8_gb300 import shard, synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    joined, offs, bases, totals = q.get(timeout=120)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert shard.layer_ranges(W["n_layers"], 2) == [(0, 3), (3, 5)]
    assert bases == [0, totals[0]]
    w = synth.WORKLOADS[W["name"]].scaled(n_layers=W["n_layers"], n_tokens=W["n_tokens"], lane_syms=W["lane_syms"])
    t, p = synth.gen_kv(w, "cpu")
    po = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib)
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    bins, _, _ = orc.calibrate(po, tn, pn)
    fr, cum = orc.build_tables(po)
    st, bs, ref_offs = orc.encode(po, fr, cum, bins, tn, pn)
    assert st == orc.OK
    assert joined == bs.tobytes()
    assert offs == ref_offs.tolist()


def test_layer_ranges_cover_everything():
    from lossless_kv_cache_fp8_gb300 import shard
    for n in (1, 7, 64):
        for world in (1, 2, 3, 8):
            r = shard.layer_ranges(n, world)
            assert r[0][0] == 0 and r[-1][1] == n and all(a[1] == b[0] for a, b in zip(r, r[1:]))
            assert max(h - l for l, h in r) - min(h - l for l, h in r) <= 1
