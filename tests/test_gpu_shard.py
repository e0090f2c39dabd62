"""Sharded encode on the CUDA library: two gloo ranks (processes) on the one
visible GPU each calibrate and encode their layer range of one cache through
libskv.so, all-gather their byte totals and place their streams; the joined
stream and lane offsets equal the one-call GPU stream of the whole cache and
the oracle's.  (Every run here has one GPU; the ranks' kernels never wait on
each other, so sharing the device is safe.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

W = dict(name="qwen3-8b-32k-fp8", n_layers=5, n_heads=2, n_tokens=1536, lane_syms=1024)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _workload():
    from lossless_kv_cache_fp8_gb300 import synth
    return synth.WORKLOADS[W["name"]].scaled(n_layers=W["n_layers"], n_heads=W["n_heads"], n_tokens=W["n_tokens"],
                                             lane_syms=W["lane_syms"])


def _rank(rank, world, port, q):
    try:
        _rank_body(rank, world, port, q)
    except BaseException:   # report at once instead of leaving the other rank in a collective
        import traceback
        q.put(("error", rank, traceback.format_exc()))
        raise


def _rank_body(rank, world, port, q):
    import datetime

    import torch.distributed as dist

    from lossless_kv_cache_fp8_gb300 import native, shard, synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    torch.cuda.set_device(0)
    w = _workload()
    lo, hi = shard.layer_ranges(w.n_layers, world)[rank]
    t, p = synth.gen_kv(w, "cuda", layers=(lo, hi))
    params = native.params_for(w)
    codec, n, base, totals = shard.encode_layer_shard(params, t, p, lo, hi)
    parts = [None] * world
    dist.all_gather_object(parts, (codec.bitstream[:n].cpu().numpy().tobytes(),
                                   codec.lane_offsets.cpu().numpy().view(np.uint64).tolist(), base))
    if rank == 0:
        shards = [shard.Shard(np.array(o, dtype=np.uint64), len(b)) for b, o, _ in parts]
        q.put(("ok", b"".join(b for b, _, _ in parts), shard.join_offsets(shards).tolist(),
               [b for _, _, b in parts], totals))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gpu_shards_join_to_one_stream(orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from lossless_kv_cache_fp8_gb300 import native, shard, synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    try:
        msg = q.get(timeout=240)
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.exitcode is None:
                pr.terminate()
                pr.join(timeout=10)
    assert msg[0] == "ok", f"rank {msg[1]} failed:\n{msg[2]}"
    _, joined, offs, bases, totals = msg
    assert all(pr.exitcode == 0 for pr in procs)
    assert bases == [0, totals[0]]
    w = _workload()
    # the whole cache in one call on this GPU
    t, p = synth.gen_kv(w, "cuda")
    codec = native.Codec(native.params_for(w))
    codec.calibrate(t, p)
    codec.build_tables()
    n = codec.encode(t, p)
    assert codec.check() == native.SKV_OK
    assert joined == codec.bitstream[:n].cpu().numpy().tobytes()
    assert offs == codec.lane_offsets.cpu().numpy().view(np.uint64).tolist()
    # and the oracle's
    po = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib)
    tn = t.cpu().numpy().reshape(-1).view(np.uint8)
    pn = p.cpu().numpy().reshape(-1).view(np.uint8)
    bins, _, _ = orc.calibrate(po, tn, pn)
    fr, cum = orc.build_tables(po)
    st, bs, ref_offs = orc.encode(po, fr, cum, bins, tn, pn)
    assert st == orc.OK
    assert joined == bs.tobytes() and offs == ref_offs.tolist()
