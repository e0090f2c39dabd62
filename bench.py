"""Benchmark: speculative KV coding round trip on one GB300.

One step = the whole hot path over one cache: calibrate (per-channel Laplace
scales), build tables, encode (rANS lanes, scan, pack), decode (fused
reconstruction).  Inputs are resident in HBM before the timed region; the
128K-token Qwen3-32B-shaped FP8 cache (2 x 17.2 GB) is far larger than L2, so no
flush is needed between steps.

Prints one JSON line.  ``value`` = raw target-cache bytes per step / step time
(GB/s, whole job).  ``e2e`` repeats the step through the same C ABI with the
inputs copied from pinned host memory and the bitstream copied back inside the
timed region.  ``--impl reference`` times the CPU oracle (the reference arm of
this method) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV codec GB/s (raw KV in) enc/dec, Qwen3-32B shape 128K, % of HBM peak; ratio"
DEFAULT_WORKLOAD = "qwen3-32b-128k-fp8"


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def kernel_source_hash():
    import hashlib
    src = os.path.join(ROOT, "lossless_kv_cache_fp8_gb300", "csrc", "skv.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def profile_fields(kernel: str):
    """the markers of the committed ncu summary of `kernel`, or {} when it is
    missing or was taken from a different kernel source"""
    path = os.path.join(ROOT, "profiles", f"{kernel}_fp8_qwen3-32b-8layers.md")
    try:
        txt = open(path).read()
    except OSError:
        return {}
    fields = {}
    for line in txt.splitlines():
        if line.startswith("<!-- ") and "=" in line:
            k, v = line[5:].rstrip(" ->").split("=", 1)
            fields[k.strip()] = v.strip()
    return fields if fields.get("source_sha256") == kernel_source_hash() else {}


def profiled_traffic(kernel: str, layers_full: int):
    """DRAM bytes per full-size launch of `kernel` from the committed ncu summary, or
    None when the summary is missing or was taken from a different kernel source."""
    fields = profile_fields(kernel)
    if not fields:
        return None
    try:
        per = float(fields["dram_bytes_per_launch"]) * layers_full / float(fields["layers"])
    except (KeyError, ValueError):
        return None
    return per


def hbm_peak():
    pk = peaks()
    if pk and pk.get("hbm_gbs"):
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region"""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# reference arm: the CPU oracle on a bounded sample of the workload
# ------------------------------------------------------------------------------------------
COEF_SAMPLE_TOKENS = 256   # sample unit of a coefficient stream (a block of whole tokens)


def sample_units(w):
    """sample units of the workload: (layer, kv, head) slices of a KV cache, blocks of
    COEF_SAMPLE_TOKENS tokens of a coefficient stream"""
    from lossless_kv_cache_fp8_gb300 import synth
    if w.dtype == synth.COEF:
        return max(1, w.n_tokens // COEF_SAMPLE_TOKENS)
    return w.n_layers * w.n_kv * w.n_heads


def sample_label(w, n):
    from lossless_kv_cache_fp8_gb300 import synth
    if w.dtype == synth.COEF:
        return f"first {n} of {sample_units(w)} blocks of {COEF_SAMPLE_TOKENS} tokens"
    return f"first {n} of {sample_units(w)} (layer,kv,head) slices"


def oracle_sample(w, n: int):
    """the first n sample units of the workload, generated on the CPU: a dict with the
    raw target bits, the prediction (the predictor cache, or the means mu) and, for a
    coefficient stream, beta and the sample's token count"""
    from lossless_kv_cache_fp8_gb300 import synth
    if w.dtype == synth.COEF:
        q, mu, beta = synth.gen_coef(w, "cpu")
        rows = min(w.n_tokens, n * COEF_SAMPLE_TOKENS)
        return {"target": q[:rows].contiguous().reshape(-1).numpy(),
                "pred": mu[:rows].contiguous().reshape(-1).numpy(), "beta": beta.numpy(), "rows": rows}
    per_layer = w.n_kv * w.n_heads
    n_layers = (n + per_layer - 1) // per_layer
    t, p = synth.gen_kv(w, "cpu", layers=(0, n_layers))
    sp = w.n_tokens * w.head_dim
    t = t.reshape(-1)[: n * sp].numpy()
    p = p.reshape(-1)[: n * sp].numpy()
    if w.dtype != synth.FP8:
        t, p = t.view("uint16"), p.view("uint16")
    return {"target": t, "pred": p}


def run_oracle_round_trip(w, s, n):
    """calibrate + tables + encode + decode of the sample s (n units) with the oracle;
    returns seconds and the stream's bytes"""
    import numpy as np
    import oracle
    from lossless_kv_cache_fp8_gb300 import synth
    oracle.build()
    t, p = s["target"], s["pred"]
    if w.dtype == synth.COEF:
        po = oracle.coef_params(s["rows"], w.n_coef, w.lane_syms)
    else:   # n slices as a cache of n heads
        po = oracle.kv_params(w.dtype, 1, 1, n, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib)
    t0 = time.perf_counter()
    if w.dtype == synth.COEF:
        bins, _, _ = oracle.calibrate(po, None, s["beta"], want_sum=False)
    else:
        bins, _, _ = oracle.calibrate(po, t, p, want_sum=False)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, t, p)
    st2, out = oracle.decode(po, fr, cum, bins, bs, offs, p, t.dtype)
    dt = time.perf_counter() - t0
    assert st == oracle.OK and st2 == oracle.OK and np.array_equal(out, t)
    return dt, bs.size


def cpu_baseline(w, target_seconds=12.0):
    """oracle round trip on the first units of the workload, about target_seconds of CPU"""
    s = oracle_sample(w, 1)
    dt1, _ = run_oracle_round_trip(w, s, 1)
    n = max(1, min(sample_units(w), int(target_seconds / max(dt1, 1e-3))))
    if n > 1:
        s = oracle_sample(w, n)
        dt, _ = run_oracle_round_trip(w, s, n)
    else:
        dt = dt1
    raw = s["target"].nbytes
    return {"value": raw / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{sample_label(w, n)} ({raw / 1e6:.1f} MB raw), "
                      f"single-threaded calibrate+tables+encode+decode"}


def main_reference(args):
    from lossless_kv_cache_fp8_gb300 import synth
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    n = max(1, min(args.ref_slices, sample_units(w)))
    s = oracle_sample(w, n)
    for _ in range(args.warmup):
        run_oracle_round_trip(w, s, n)
    times = []
    for _ in range(args.steps):
        dt, _ = run_oracle_round_trip(w, s, n)
        times.append(dt)
    total = sum(times)
    raw = s["target"].nbytes
    v = raw * len(times) / total / 1e9
    sample = f"{sample_label(w, n)} ({raw / 1e6:.1f} MB raw) per step, single-threaded"
    dtype = {synth.FP8: "u8", synth.BF16: "u16", synth.COEF: "i16"}[w.dtype]
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype, "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------
def main_ours(args):
    import torch
    from lossless_kv_cache_fp8_gb300 import build as libbuild
    from lossless_kv_cache_fp8_gb300 import native, synth

    from lossless_kv_cache_fp8_gb300 import shard
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    libbuild.build()
    w_full = synth.WORKLOADS[args.workload]
    if args.layers:
        w_full = w_full.scaled(n_layers=args.layers)
    if args.lane_syms:
        w_full = w_full.scaled(lane_syms=args.lane_syms)
    # N ranks: a KV cache is split by layers (each rank codes its layer range of
    # the one cache; the streams join after an all-gather of the byte totals);
    # a coefficient stream is one slice, so each rank codes its own copy
    split = world > 1 and w_full.dtype != synth.COEF
    lo, hi = shard.layer_ranges(w_full.n_layers, world)[rank] if split else (0, w_full.n_layers)
    w = w_full.scaled(n_layers=hi - lo) if split else w_full
    p = native.params_for(w, model=args.model)
    sz = native.sizes(p)
    stream = torch.cuda.current_stream(dev)

    # inputs resident in HBM before the timed region
    if split:
        tgt, prd = synth.gen_kv(w_full, dev, layers=(lo, hi))
        cal = prd
    else:
        tgt, prd, cal = synth.gen_workload(w, dev)
    torch.cuda.empty_cache()
    codec = native.Codec(p, device=dev, bitstream_capacity=int(w.raw_bytes * args.cap_frac))
    out = torch.empty_like(tgt)
    torch.cuda.synchronize()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        codec.calibrate(None if w.dtype == synth.COEF else tgt, cal)
        if ev:
            ev[1].record(stream)
        codec.build_tables()
        if ev:
            ev[2].record(stream)
        codec.encode(tgt, prd, want_total=False)
        if ev:
            ev[3].record(stream)
        codec.decode(prd, out, n_bytes=step.n_bytes)   # same stream every step (deterministic)
        if ev:
            ev[4].record(stream)

    # first pass: sizes, correctness
    codec.calibrate(None if w.dtype == synth.COEF else tgt, cal)
    codec.build_tables()
    total = codec.encode(tgt, prd, want_total=True)
    st = codec.check()
    assert st == native.SKV_OK, native.status_string(st)
    step.n_bytes = total
    codec.decode(prd, out, n_bytes=total)
    assert codec.check() == native.SKV_OK and torch.equal(out, tgt), "round trip failed"

    for _ in range(args.warmup):
        step(ev=[torch.cuda.Event(enable_timing=True) for _ in range(5)])
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(args.steps):
            step(ev=evs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    st = codec.check()
    assert st == native.SKV_OK, native.status_string(st)
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms, world, dev)
    phase = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
             for i, name in enumerate(["calibrate", "build_tables", "encode", "decode"])}

    peak, peak_kind = hbm_peak()
    raw = w.raw_bytes
    pred_bytes = w.n_positions * (4 if w.dtype == synth.COEF else w.elem_bytes)
    lanes = sz["lanes"]
    enc_bytes = raw + pred_bytes + total + 8 * (lanes + 1)           # in: both caches; out: stream + offsets
    dec_bytes = pred_bytes + total + 8 * (lanes + 1) + raw           # in: pred + stream + offsets; out: target
    enc_gbs = enc_bytes / phase["encode"] / 1e6
    dec_gbs = dec_bytes / phase["decode"] / 1e6
    dominant = "decode" if phase["decode"] >= phase["encode"] else "encode"
    achieved = dec_gbs if dominant == "decode" else enc_gbs
    kname = "k_decode_kv" if dominant == "decode" else "k_encode_kv"
    # the committed ncu summaries are of the per-channel-scale kernels on this cache shape
    profiled = w.name == "qwen3-32b-128k-fp8" and args.model == 0
    traffic = profiled_traffic(kname, w.n_layers) if profiled else None
    pf = profile_fields(kname) if profiled else {}
    stored = total + 4 * lanes + sz["channels"] + 64
    if split:
        # the joined stream: one all-gather of the byte totals
        totals = shard.gather_totals(total)
        stored = sum(totals) + 4 * native.sizes(native.params_for(w_full, model=args.model))["lanes"] + \
            native.sizes(native.params_for(w_full, model=args.model))["channels"] + 64
        value = w_full.raw_bytes / (ms * 1e-3) / 1e9
    else:
        value = raw * world / (ms * 1e-3) / 1e9

    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None, "dtype": "u8" if w.dtype == synth.FP8 else ("u16" if w.dtype == synth.BF16 else "i16"),
        "data": "synthetic",
        "config": {"workload": w.name, "shape": list(w_full.shape()), "lane_syms": w.lane_syms,
                   "parallelism": f"layers split over {world} GPUs" if split else
                   ("one GPU" if world == 1 else f"{world} independent replicas"),
                   "residual_model": ["per-channel scale", "exponent-normalised scale"][args.model],
                   "l2": "inputs larger than L2 (no flush)",
                   "step": "calibrate + build_tables + encode + decode"},
        "phases_ms": phase,
        "encode_raw_gbs": raw / phase["encode"] / 1e6, "decode_raw_gbs": raw / phase["decode"] / 1e6,
        "encode_total_gbs": enc_gbs, "decode_total_gbs": dec_gbs,
        "encode_hbm_frac": enc_gbs / peak, "decode_hbm_frac": dec_gbs / peak,
        "ratio": (w_full.raw_bytes if split else raw) / stored, "bitstream_bytes": total,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic,
                     "inst_per_position": float(pf["warp_inst_per_warp_position"])
                     if "warp_inst_per_warp_position" in pf else None,
                     "algorithmic_bytes": dec_bytes if dominant == "decode" else enc_bytes,
                     "note": "per-call CUDA events; the encode call is one kernel after a memset of its "
                             "look-back state, the decode call is one kernel"},
        # our kernels per step: calibrate, build_tables, encode (KV: one kernel; COEF: code,
        # three scan kernels, pack), decode
        "gpu_launches": (4 if w.dtype != synth.COEF else 8) * args.steps,
        "clocks": clk.summary(),
    }
    if args.paged and w.dtype != synth.COEF:
        res["paged"] = paged_run(args, w, codec, tgt, prd, stream, total, peak)
    if args.checkerboard and w.dtype == synth.COEF:
        res["checkerboard"] = checkerboard_run(args, w, stream, dev)
    if args.e2e and world >= 1:
        res["e2e"] = e2e(args, w, codec, tgt, prd, cal, out, stream, dev, total)
        if res["e2e"].get("value") is not None and world > 1:
            e_ms = max_over_ranks(res["e2e"]["ms_per_step"], world, dev)
            res["e2e"]["ms_per_step"] = e_ms
            res["e2e"]["value"] = (w_full.raw_bytes if split else raw * world) / (e_ms * 1e-3) / 1e9
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)


def e2e(args, w, codec, tgt, prd, cal, out, stream, dev, total):
    """The same round trip through the C ABI from host buffers.  KV caches:
    skv_encode_host (pinned target + prediction in, stream + lane offsets out)
    then skv_decode_host (stream + offsets + prediction in, decoded target out),
    each coding layer groups with the copies overlapped on three streams inside
    the library; the stream, offsets and decoded cache are checked against the
    one-call results.  Coefficient streams are copied in, coded and copied back
    in sequence."""
    import torch
    from lossless_kv_cache_fp8_gb300 import native, pipeline, synth
    try:
        # page-locked host buffers backed by huge pages (see pipeline.pinned_empty)
        h_t = pipeline.pinned_empty(tgt.shape, tgt.dtype)
        h_p = pipeline.pinned_empty(prd.shape, prd.dtype)
        h_bs = pipeline.pinned_empty((int(total * 1.05) + 4096,), torch.uint8)
        h_out = pipeline.pinned_empty(tgt.shape, tgt.dtype) if w.dtype != synth.COEF else None
    except RuntimeError as e:
        return {"value": None, "unit": "GB/s", "error": f"pinned host allocation failed: {e}"[:200]}
    h_t.copy_(tgt)
    h_p.copy_(prd)
    h_off = torch.empty(codec.lane_offsets.shape, dtype=torch.int64, pin_memory=True)
    torch.cuda.synchronize()
    kv = w.dtype != synth.COEF
    pipe = None
    if kv:
        groups = max(1, min(16, w.n_layers))
        pipe = pipeline.HostPipeline(codec.p, group_layers=-(-w.n_layers // groups), device=dev,
                                     cap_frac=args.cap_frac)
    times, t_enc, t_dec = [], [], []
    nb = 0
    for k in range(args.warmup + max(1, args.e2e_steps)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if kv:
            n = pipe.encode(h_t, h_p, h_bs, h_off)
            t1 = time.perf_counter()
            pipe.decode(h_bs, n, h_off, h_p, h_out)
        else:
            tgt.copy_(h_t, non_blocking=True)
            prd.copy_(h_p, non_blocking=True)
            codec.calibrate(None, cal)
            codec.build_tables()
            n = codec.encode(tgt, prd, want_total=True)
            h_bs[:n].copy_(codec.bitstream[:n], non_blocking=True)
            h_off.copy_(codec.lane_offsets, non_blocking=True)
            torch.cuda.synchronize()
            t1 = time.perf_counter()
            codec.decode(prd, out, n_bytes=n)
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        if k >= args.warmup:
            times.append((t2 - t0) * 1e3)
            t_enc.append((t1 - t0) * 1e3)
            t_dec.append((t2 - t1) * 1e3)
        nb = n
    res = {}
    if kv:
        assert nb == total and torch.equal(h_bs[:nb], codec.bitstream[:nb].cpu())
        assert torch.equal(h_off, codec.lane_offsets.cpu())
        assert torch.equal(h_out, tgt.cpu())
        res["pipeline"] = {"layer_groups": len(pipe.groups), "streams": 3, "calls": "skv_encode_host, skv_decode_host",
                           "check": "stream, offsets and decoded cache equal the one-call results"}
        h2d = 2 * w.raw_bytes + nb + h_off.numel() * 8 + w.raw_bytes   # encode: target + prediction; decode: stream + offsets + prediction
        d2h = nb + h_off.numel() * 8 + w.raw_bytes                       # encode: stream + offsets; decode: target
    else:
        assert torch.equal(out, tgt)
        h2d = h_t.numel() * h_t.element_size() + h_p.numel() * h_p.element_size()
        d2h = nb + h_off.numel() * 8
    ms = statistics.mean(times)
    return {"value": w.raw_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "encode_ms": statistics.mean(t_enc),
            "decode_ms": statistics.mean(t_dec), "steps": len(times),
            "timing": "host wall clock around the synchronous calls (copies included)", **res}


def paged_run(args, w, codec, tgt, prd, stream, total, peak):
    """encode / decode the same cache held in paged pools (random block table,
    args.paged tokens per block); the stream must equal the dense one"""
    import torch
    from lossless_kv_cache_fp8_gb300 import native, synth
    B = args.paged
    tp, pp, table, n_blocks = synth.to_paged(tgt, prd, B, seed=1)
    lay = native.paged_layout(table, n_blocks, B)
    p = codec.p
    bs = torch.empty_like(codec.bitstream)
    off = torch.empty_like(codec.lane_offsets)
    outp = torch.zeros_like(tp)
    status = torch.zeros(4, dtype=torch.int32, device=tgt.device)

    def enc():
        st, _ = native.skv_encode_paged(p, lay, tp, pp, codec.tables, codec.bins, bs, codec.cap, off,
                                        codec.workspace, codec.workspace.numel(), status, want_total=False)
        assert st == native.SKV_OK

    def dec():
        assert native.skv_decode_paged(p, lay, bs, total, off, pp, codec.tables, codec.bins, outp,
                                       status) == native.SKV_OK

    ms = {}
    for name, fn in (("encode", enc), ("decode", dec)):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / args.steps
        assert native.skv_read_status(status) == native.SKV_OK
    assert torch.equal(bs[:total], codec.bitstream[:total]) and torch.equal(off, codec.lane_offsets)
    assert torch.equal(outp, tp)
    raw = w.raw_bytes
    moved = 2 * raw + total + 8 * off.numel()
    return {"block_tokens": B, "n_blocks": n_blocks, "encode_ms": ms["encode"], "decode_ms": ms["decode"],
            "encode_hbm_frac": moved / ms["encode"] / 1e6 / peak, "decode_hbm_frac": moved / ms["decode"] / 1e6 / peak,
            "check": "stream, offsets and decoded pool equal the dense call"}


def checkerboard_run(args, w, stream, dev):
    """The coefficient stream split by token parity with the checkerboard context:
    even rows coded with their means, odd rows with the context-shifted means
    (skv_ctx_means: two tcgen05 tensor-core products), the two parities on two
    streams; decode = even rows, context, odd rows.  Reports the context call's tensor throughput and the ratio
    against coding the odd rows with their token-conditioned means alone."""
    import torch
    from lossless_kv_cache_fp8_gb300 import native, synth
    qe, qo, me, mo, beta, V, U = synth.gen_coef_checkerboard(w, dev)
    s1, s2 = synth.CTX_SHIFT1, synth.CTX_SHIFT2
    C, n_e, n_o, R = qe.shape[1], qe.shape[0], qo.shape[0], V.shape[0]
    cmap = native.ctx_map(V, U, s1, s2)
    scratch = torch.empty(native.skv_ctx_scratch_bytes(n_o, C, R), dtype=torch.uint8, device=dev)
    mo2 = torch.empty_like(mo)
    ce = native.Codec(native.coef_params(n_e, C, w.lane_syms), device=dev)
    co = native.Codec(native.coef_params(n_o, C, w.lane_syms), device=dev)
    for c in (ce, co):
        c.calibrate(None, beta)
        c.build_tables()

    ctx_status = torch.zeros(4, dtype=torch.int32, device=dev)

    def ctx(q_even):
        assert native.skv_ctx_means(cmap, q_even, n_e, mo, n_o, C, mo2, scratch, ctx_status) == native.SKV_OK

    ctx(qe)
    ne, no = ce.encode(qe, me), co.encode(qo, mo2)
    co_plain = native.Codec(native.coef_params(n_o, C, w.lane_syms), device=dev)
    co_plain.calibrate(None, beta)
    co_plain.build_tables()
    n_plain = co_plain.encode(qo, mo)
    del co_plain
    qe_d, qo_d = torch.empty_like(qe), torch.empty_like(qo)

    # the two parities encode concurrently: the odd rows' context needs only q_even
    side = torch.cuda.Stream(dev)

    def enc():
        side.wait_stream(stream)
        ce.encode(qe, me, want_total=False, stream=side)
        ctx(qe)
        co.encode(qo, mo2, want_total=False)
        stream.wait_stream(side)

    def dec():
        ce.decode(me, qe_d)
        ctx(qe_d)
        co.decode(mo2, qo_d)

    ms = {}
    for name, fn in (("context", lambda: ctx(qe)), ("encode", enc), ("decode", dec)):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / args.steps
    assert ce.check() == native.SKV_OK and co.check() == native.SKV_OK
    assert native.skv_read_status(ctx_status) == native.SKV_OK
    assert torch.equal(qe_d, qe) and torch.equal(qo_d, qo)
    raw = (n_e + n_o) * C * 2
    flops = 2.0 * n_o * C * R * 2
    pk = peaks() or {}
    tpeak = float(pk.get("bf16_tflops") or 1900.0)
    tf = flops / ms["context"] / 1e9
    return {"rows": [n_e, n_o], "rank": R, "context_ms": ms["context"], "encode_ms": ms["encode"],
            "decode_ms": ms["decode"], "context_tflops": tf, "context_tensor_frac": tf / tpeak,
            "ratio": raw / (ne + no), "odd_rows_bytes": no, "odd_rows_bytes_without_context": n_plain,
            "check": "both parities decode to the input; context bit-exact with the oracle in tests"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--lane-syms", type=int, default=0, help="override the positions per lane of the workload")
    ap.add_argument("--cap-frac", type=float, default=0.6, help="bitstream buffer / raw bytes")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--paged", type=int, default=0, help="also time paged pools with this many tokens per block")
    ap.add_argument("--checkerboard", action="store_true",
                    help="coefficient workloads: also time the checkerboard context (two-pass) coding")
    ap.add_argument("--model", type=int, default=0, choices=[0, 1],
                    help="residual model: 0 per-channel scale (default), 1 exponent-normalised (FP8)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-slices", type=int, default=2,
                    help="reference arm: sample units per step ((layer,kv,head) slices of a KV cache, "
                         "blocks of 256 tokens of a coefficient stream)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
