"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact comparisons (integer path): calibration bins / sums / histograms, every
table's frequencies and cumulative frequencies, bitstream bytes, lane offsets and
decoded caches.  Small shapes compare everything in one oracle call; the large
full-size workloads compare every chunk with the oracle coding that chunk from its
own data (in host threads), plus decode(encode(x)) == x on the whole cache.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_kv_cache_fp8_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nat():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from lossless_kv_cache_fp8_gb300 import native
    return native


def oparams(w):
    if w.dtype == synth.COEF:
        return oracle.coef_params(w.n_tokens, w.n_coef, w.lane_syms)
    return oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                            w.n_calib)


def host_bits(x: torch.Tensor) -> np.ndarray:
    a = x.detach().cpu().numpy().reshape(-1)
    if a.dtype == np.int16:
        return a.view(np.uint16)
    return a


def table_arrays(nat, codec):
    blob = codec.tables.cpu().numpy()
    nt = codec.sz["tables"]
    blob = blob[: nt * nat.SKV_TABLE_STRIDE].reshape(nt, nat.SKV_TABLE_STRIDE)
    fr = blob[:, nat.SKV_TABLE_FREQ_OFF:nat.SKV_TABLE_FREQ_OFF + 512].copy().view(np.uint16)
    cum = blob[:, nat.SKV_TABLE_CUM_OFF:nat.SKV_TABLE_CUM_OFF + 514].copy().view(np.uint16)
    return blob, fr, cum


def run_gpu(nat, w, t, p, c, cap=None):
    codec = nat.Codec(nat.params_for(w), bitstream_capacity=cap)
    codec.calibrate(None if w.dtype == synth.COEF else t, c)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    out = torch.empty_like(t)
    codec.decode(p, out)
    assert codec.check() == nat.SKV_OK
    return codec, total, out


SMALL = [
    synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=2, n_tokens=512),
    synth.WORKLOADS["qwen3-0.6b-8k-bf16"].scaled(n_layers=1, n_tokens=384),
    synth.WORKLOADS["qwen3-8b-32k-fp8"].scaled(n_layers=1, n_heads=2, n_tokens=1024, lane_syms=256),
    synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=64, n_coef=256, lane_syms=64),
    # ragged: tokens not a multiple of the chunk, fewer tokens than calibration, odd head dims
    synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_heads=3, n_tokens=77, head_dim=32, lane_syms=48),
    synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_heads=1, n_tokens=1000, head_dim=16, lane_syms=16),
    synth.WORKLOADS["qwen3-0.6b-8k-bf16"].scaled(n_layers=1, n_heads=1, n_tokens=1, head_dim=16, lane_syms=8),
    synth.WORKLOADS["qwen3-0.6b-8k-bf16"].scaled(n_layers=2, n_heads=2, n_tokens=300, head_dim=256, lane_syms=40),
    synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=7, n_coef=37, lane_syms=24),
    synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=33, n_coef=3, lane_syms=8),
]


def full_compare(nat, w):
    t, p, c = synth.gen_workload(w, "cpu")
    td, pd, cd = t.cuda(), p.cuda(), c.cuda()
    codec, total, out = run_gpu(nat, w, td, pd, cd)
    assert torch.equal(out, td)
    po = oparams(w)
    tn, pn, cn = host_bits(t), host_bits(p), c.numpy().reshape(-1) if w.dtype == synth.COEF else host_bits(c)
    if w.dtype == synth.COEF:
        tn = t.numpy().reshape(-1)
        pn = p.numpy().reshape(-1)
        bins, _, _ = oracle.calibrate(po, None, cn)
    else:
        bins, sums, _ = oracle.calibrate(po, tn, cn)
    nch = bins.size
    assert np.array_equal(codec.bins[:nch].cpu().numpy(), bins)
    fr, cum = oracle.build_tables(po)
    _, gfr, gcum = table_arrays(nat, codec)
    assert np.array_equal(gfr, fr) and np.array_equal(gcum, cum)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    assert total == bs.size
    assert np.array_equal(codec.lane_offsets.cpu().numpy().astype(np.uint64), offs)
    assert np.array_equal(codec.bitstream[:total].cpu().numpy(), bs)
    return codec


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"{w.name}-L{w.n_layers}H{w.n_heads}T{w.n_tokens}D{w.head_dim}K{w.lane_syms}")
def test_small_bit_exact(nat, w):
    full_compare(nat, w)


@pytest.mark.parametrize("off", [2, 6, 14])
def test_stream_at_unaligned_addresses(nat, off):
    """The stream need only be 2-byte aligned: written at an address 2, 6 or 14
    bytes past a 16-byte boundary it holds the same bytes and offsets, and
    nothing outside it is touched.  Lanes of 16 positions give about four chunks
    per warp, so both chunk copies run (lane by lane before the last wave,
    through the staging slots in it)."""
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=4, lane_syms=16)
    codec = full_compare(nat, w)   # aligned stream == the oracle's
    t, p, _ = synth.gen_workload(w, "cpu")   # the inputs full_compare coded
    t, p = t.cuda(), p.cuda()
    total = codec.n_bytes
    ref, ref_off = codec.bitstream[:total].clone(), codec.lane_offsets.clone()
    buf = torch.full((codec.cap + 32,), 0xCD, dtype=torch.uint8, device="cuda")
    view = buf[off:off + codec.cap]
    codec.lane_offsets.fill_(-1)
    st, tot = nat.skv_encode(codec.p, t, p, codec.tables, codec.bins, view, codec.cap, codec.lane_offsets,
                             codec.workspace, codec.workspace.numel(), codec.status, want_total=True)
    assert st == nat.SKV_OK and codec.check() == nat.SKV_OK and tot == total
    assert torch.equal(view[:total], ref) and torch.equal(codec.lane_offsets, ref_off)
    assert bool((buf[:off] == 0xCD).all()) and bool((buf[off + total:] == 0xCD).all())


def test_calibration_sums_and_histograms(nat):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_tokens=600)
    t, p, _ = synth.gen_workload(w, "cpu")
    po = oparams(w)
    bins, sums, hist = oracle.calibrate(po, host_bits(t), host_bits(p), want_sum=True, want_hist=True)
    codec = nat.Codec(nat.params_for(w))
    s_d = torch.zeros(bins.size, dtype=torch.int32, device="cuda")
    h_d = torch.zeros(bins.size * 256, dtype=torch.int32, device="cuda")
    codec.calibrate(t.cuda(), p.cuda(), sum_abs=s_d, hist=h_d)
    torch.cuda.synchronize()
    assert np.array_equal(codec.bins[: bins.size].cpu().numpy(), bins)
    assert np.array_equal(s_d.cpu().numpy().view(np.uint32), sums)
    assert np.array_equal(h_d.cpu().numpy().view(np.uint32).reshape(-1, 256), hist)


@pytest.mark.parametrize("kind", ["kv", "coef"])
def test_table_blob_structures(nat, kind):
    """encoder reciprocals, slot->symbol tables and decoder entries are consistent
    with the frequencies (checked on the host from their definitions)"""
    p = nat.kv_params(1, 1, 2, 1, 128, 16, 16) if kind == "kv" else nat.coef_params(4, 16, 8)
    codec = nat.Codec(p)
    codec.build_tables()
    torch.cuda.synchronize()
    blob, fr, cum = table_arrays(nat, codec)
    for t in range(blob.shape[0]):
        f = fr[t].astype(np.int64)
        c = cum[t].astype(np.int64)
        enc = blob[t, nat.SKV_TABLE_ENC_OFF:nat.SKV_TABLE_ENC_OFF + 2048].copy().view(np.uint32).reshape(256, 2)
        for i in range(256):
            fi = int(f[i])
            w = int(enc[i, 1])
            sh, h = w & 31, (w >> 7) & 1
            assert w >> 20 == fi and (w >> 8) & 0xFFF == int(c[i]) and (w >> 5) & 3 == 0
            # s = ceil(log2 fr) and the reciprocal's top bit is 2^32
            assert h == 1 and (1 << sh) >= fi and (sh == 0 or (1 << (sh - 1)) < fi)
            k = 1 << (32 + sh)
            m = (h << 32) | int(enc[i, 0])
            assert m == -(-k // fi)
            # floor(x/fr) = floor(x m / 2^(32+s)) for every x < fr 2^20 and x m < 2^64
            x1 = fi * (1 << 20) - 1
            assert x1 * (m * fi - k) < k and x1 * m < (1 << 64)
        dec = blob[t, nat.SKV_TABLE_DEC_OFF:nat.SKV_TABLE_DEC_OFF + 1024].copy().view(np.uint32)
        # fr in the lower half, -cum as a signed upper half
        assert np.array_equal(dec & 0xFFFF, f.astype(np.uint32))
        assert np.array_equal(dec.view(np.int32) >> 16, -c[:256].astype(np.int32))
        lut = blob[t, nat.SKV_TABLE_LUT_OFF:nat.SKV_TABLE_LUT_OFF + 4096]
        assert np.array_equal(lut, np.repeat(np.arange(256), f).astype(np.uint8))
    if kind == "coef":
        # slot entries after the tables: symbol | fr << 8 | (slot - cum) << 20
        nt = blob.shape[0]
        raw = codec.tables.cpu().numpy()
        assert raw.size == nt * (nat.SKV_TABLE_STRIDE + nat.SKV_TABLE_SLOT_BYTES)
        se = raw[nt * nat.SKV_TABLE_STRIDE:].copy().view(np.uint32).reshape(nt, 4096).astype(np.int64)
        slots = np.arange(4096)
        for t in range(nt):
            sym = np.repeat(np.arange(256), fr[t].astype(np.int64))
            want = sym | (fr[t].astype(np.int64)[sym] << 8) | ((slots - cum[t].astype(np.int64)[sym]) << 20)
            assert np.array_equal(se[t], want), t


FULL_EXACT = ["qwen3-0.6b-1k-fp8", "hybrid-coef-32k-x2048"]


@pytest.mark.parametrize("name", FULL_EXACT)
def test_full_size_bit_exact(nat, name):
    """whole workloads the oracle codes in seconds: every byte compared"""
    full_compare(nat, synth.WORKLOADS[name])


def every_chunk_compare(nat, w, model=0):
    """generate on the GPU, code the whole cache there, then check every slice's
    bins and every chunk's words and lane lengths against the oracle coding that
    chunk from its own data (host threads: the oracle's C calls release the GIL)"""
    import concurrent.futures as cf
    import os
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(nat.params_for(w, model=model), bitstream_capacity=w.raw_bytes)
    codec.calibrate(t, c)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    out = torch.empty_like(t)
    codec.decode(p, out)
    assert codec.check() == nat.SKV_OK
    assert torch.equal(out, t)
    del out
    po = oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                          w.n_calib, model=model)
    g = oracle.geometry(po)
    fr, cum = oracle.build_tables(po)
    _, gfr, gcum = table_arrays(nat, codec)
    assert np.array_equal(gfr, fr) and np.array_equal(gcum, cum)
    tn, pn = host_bits(t), host_bits(p)
    del t, p, c
    torch.cuda.empty_cache()
    assert total % 2 == 0
    bs = codec.bitstream[:total].cpu().numpy().view(np.uint16)
    offs = codec.lane_offsets.cpu().numpy().astype(np.int64)
    assert offs[0] == 0 and offs[-1] == total and np.all(np.diff(offs) >= 4)
    gbins = codec.bins[: g["n_channels"]].cpu().numpy()
    sp, cps, cs, D = g["slice_positions"], g["chunks_per_slice"], 32 * w.lane_syms, w.head_dim
    ncal = min(w.n_calib, w.n_tokens)
    po1 = oracle.kv_params(w.dtype, 1, 1, 1, D, ncal, w.lane_syms, w.n_calib, model=model)

    def slice_job(sl):
        s0 = sl * sp
        b1, _, _ = oracle.calibrate(po1, tn[s0:s0 + ncal * D], pn[s0:s0 + ncal * D])
        if not np.array_equal(gbins[sl * D:(sl + 1) * D], b1):
            return f"bins of slice {sl}"
        for k in range(cps):
            ch = sl * cps + k
            first, n_pos = s0 + k * cs, min(cs, sp - k * cs)
            words, lw = oracle.encode_chunk(po, ch, fr, cum, gbins, tn[first:first + n_pos], pn[first:first + n_pos])
            a, b = offs[32 * ch], offs[32 * ch + 32]
            if not np.array_equal(bs[a // 2:b // 2], words):
                return f"chunk {ch}"
            if not np.array_equal(np.diff(offs[32 * ch:32 * ch + 33]) // 2, lw.astype(np.int64)):
                return f"lane lengths of chunk {ch}"
        return None

    with cf.ThreadPoolExecutor(os.cpu_count() or 4) as ex:
        errs = [e for e in ex.map(slice_job, range(g["n_chunks"] // cps)) if e]
    assert not errs, errs[:5]
    return codec, total


@pytest.mark.parametrize("name", ["qwen3-0.6b-8k-bf16", "qwen3-8b-32k-fp8", "qwen3-32b-128k-fp8"])
def test_full_size_every_chunk(nat, name):
    """the three large workloads at full size: every byte of the stream and every
    lane offset against the oracle (chunk by chunk), every slice's bins, and the
    decoded cache equal to the input"""
    w = synth.WORKLOADS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 2 * w.raw_bytes + w.raw_bytes + nat.sizes(nat.params_for(w))["workspace"] + w.raw_bytes
    if need > free:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")
    codec, total = every_chunk_compare(nat, w)
    ratio = w.raw_bytes / (total + 4 * codec.sz["lanes"] + codec.sz["channels"] + 64)
    print(f"{name}: {w.raw_bytes / 1e9:.2f} GB -> {total / 1e9:.3f} GB, ratio {ratio:.3f}")
    del codec
    torch.cuda.empty_cache()


def test_full_size_every_chunk_exponent_model(nat):
    """the 128K Qwen3-32B-shaped FP8 cache with the exponent residual model: every
    chunk and every slice's base bins against the oracle"""
    w = synth.WORKLOADS["qwen3-32b-128k-fp8"]
    free, _ = torch.cuda.mem_get_info()
    need = 2 * w.raw_bytes + w.raw_bytes + nat.sizes(nat.params_for(w))["workspace"] + w.raw_bytes
    if need > free:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")
    codec, total = every_chunk_compare(nat, w, model=nat.SKV_MODEL_EXPONENT)
    print(f"exponent model: {w.raw_bytes / 1e9:.2f} GB -> {total / 1e9:.3f} GB")
    del codec
    torch.cuda.empty_cache()


def test_oracle_decodes_gpu_stream(nat):
    w = SMALL[1]
    codec = full_compare(nat, w)
    t, p, c = synth.gen_workload(w, "cpu")
    po = oparams(w)
    bins = codec.bins[: oracle.geometry(po)["n_channels"]].cpu().numpy()
    fr, cum = oracle.build_tables(po)
    bs = codec.bitstream[: codec.n_bytes].cpu().numpy()
    st, out = oracle.decode(po, fr, cum, bins, bs, codec.lane_offsets.cpu().numpy().astype(np.uint64),
                            host_bits(p), np.uint16)
    assert st == oracle.OK and np.array_equal(out, host_bits(t))


def test_deterministic(nat):
    w = SMALL[0]
    t, p, c = synth.gen_workload(w, "cuda")
    c1, n1, _ = run_gpu(nat, w, t, p, c)
    c2, n2, _ = run_gpu(nat, w, t, p, c)
    assert n1 == n2 and torch.equal(c1.bitstream[:n1], c2.bitstream[:n2])


def test_corrupt_streams_reported(nat):
    w = SMALL[0]
    t, p, c = synth.gen_workload(w, "cuda")
    codec, total, _ = run_gpu(nat, w, t, p, c)
    out = torch.empty_like(t)
    # damaged state words of one lane
    bs = codec.bitstream.clone()
    a = int(codec.lane_offsets[7])
    bs[a + 1] ^= 0x40
    codec.decode(p, out, bitstream=bs)
    assert codec.check() == nat.SKV_ERR_CORRUPT
    # stream shorter than the offsets say
    codec.decode(p, out, n_bytes=total - 2)
    assert codec.check() == nat.SKV_ERR_CORRUPT
    # offsets out of order
    lo = codec.lane_offsets.clone()
    lo[3], lo[4] = codec.lane_offsets[4].item(), codec.lane_offsets[3].item()
    codec.decode(p, out, lane_offsets=lo)
    assert codec.check() == nat.SKV_ERR_CORRUPT
    # the intact stream still decodes
    codec.decode(p, out)
    assert codec.check() == nat.SKV_OK and torch.equal(out, t)


def test_capacity(nat):
    w = SMALL[0]
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(nat.params_for(w), bitstream_capacity=64)
    codec.calibrate(t, c)
    codec.build_tables()
    st, tot = nat.skv_encode(codec.p, t, p, codec.tables, codec.bins, codec.bitstream, codec.cap,
                             codec.lane_offsets, codec.workspace, codec.workspace.numel(), codec.status)
    assert st == nat.SKV_ERR_CAPACITY and tot > 64
    st, _ = nat.skv_encode(codec.p, t, p, codec.tables, codec.bins, codec.bitstream, codec.cap,
                           codec.lane_offsets, codec.workspace, codec.workspace.numel(), codec.status,
                           want_total=False)
    assert st == nat.SKV_OK
    assert codec.check() == nat.SKV_ERR_CAPACITY


def test_argument_errors(nat):
    w = SMALL[0]
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(nat.params_for(w))
    raw = torch.empty(t.numel() + 16, dtype=torch.uint8, device="cuda")
    st = nat.skv_calibrate(codec.p, raw.data_ptr() + 1, p, codec.bins)
    assert st == nat.SKV_ERR_INVALID_ARG
    codec.calibrate(t, c)
    codec.build_tables()
    st, _ = nat.skv_encode(codec.p, t, p, codec.tables, codec.bins, codec.bitstream, codec.cap,
                           codec.lane_offsets, codec.workspace, 16, codec.status)
    assert st == nat.SKV_ERR_INVALID_ARG                  # workspace too small
    bad = codec.bins.clone()
    bad[5] = 200                                          # out-of-range bin
    st, _ = nat.skv_encode(codec.p, t, p, codec.tables, bad, codec.bitstream, codec.cap,
                           codec.lane_offsets, codec.workspace, codec.workspace.numel(), codec.status)
    assert st == nat.SKV_OK
    assert codec.check() == nat.SKV_ERR_INVALID_ARG


def test_empty(nat):
    p = nat.kv_params(1, 2, 2, 2, 128, 0, 1024)
    codec = nat.Codec(p)
    t = torch.empty(16, dtype=torch.uint8, device="cuda")
    codec.calibrate(t, t)
    codec.build_tables()
    assert codec.encode(t, t) == 0
    assert int(codec.lane_offsets[0]) == 0
    codec.decode(t, t)
    assert codec.check() == nat.SKV_OK


@pytest.mark.parametrize("n,missing", [(64, 20), (300, 0), (200, 199)])
def test_lookback_gives_up_without_hanging(nat, n, missing):
    """the encoder's chunk look-back: predecessors' prefixes are exact, a chunk that
    never publishes makes its successor time out (bounded polling) and later chunks
    fail at once; the context stays usable afterwards"""
    import time
    state = torch.zeros(n, dtype=torch.int64, device="cuda")
    excl = torch.zeros(n, dtype=torch.int64, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    assert nat.skv_selftest_lookback(state, n, missing, 2000, excl, status) == nat.SKV_OK
    st = nat.skv_read_status(status)
    dt = time.perf_counter() - t0
    e = excl.cpu().numpy().astype(np.uint64)
    for w in range(missing):
        assert int(e[w]) == w * (w + 1) // 2          # sum of totals 1..w
    for w in range(missing + 1, n):
        assert int(e[w]) == (1 << 64) - 1
    assert st == (nat.SKV_ERR_TIMEOUT if missing + 1 < n else nat.SKV_OK)
    assert dt < 10.0
    # a normal call still works afterwards
    ok = torch.zeros(n, dtype=torch.int64, device="cuda")
    assert nat.skv_selftest_lookback(ok, n, n + 5, 2000, excl, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    e = excl.cpu().numpy()
    assert all(int(e[w]) == w * (w + 1) // 2 for w in range(n))


def _adversarial(kind, dtype, n, seed):
    rng = np.random.default_rng(seed)
    if dtype == synth.FP8:
        hi, dt = 256, np.uint8
        nan, neg0, maxv = 0x7F, 0x80, 0x7E
    else:
        hi, dt = 1 << 16, np.uint16
        nan, neg0, maxv = 0x7FC0, 0x8000, 0x7F7F
    if kind == "uniform":                    # residuals everywhere: many escapes
        t, p = rng.integers(0, hi, n), rng.integers(0, hi, n)
    elif kind == "nan":                      # all NaN target, zero prediction
        t, p = np.full(n, nan), np.zeros(n, np.int64)
    elif kind == "signflip":                 # prediction = target with the sign bit flipped
        t = rng.integers(0, hi, n)
        p = t ^ (hi >> 1)
    elif kind == "extremes":                 # largest magnitudes against -0 / +0
        t = np.where(rng.random(n) < 0.5, maxv, maxv | (hi >> 1))
        p = np.where(rng.random(n) < 0.5, neg0, 0)
    else:                                    # mixture: mostly near, 1% wild
        t = rng.integers(0, hi, n)
        p = np.where(rng.random(n) < 0.01, rng.integers(0, hi, n), np.clip(t + rng.integers(-2, 3, n), 0, hi - 1))
    return t.astype(dt), p.astype(dt)


@pytest.mark.parametrize("dtype", [synth.FP8, synth.BF16])
def test_long_and_short_lanes_in_one_chunk(nat, dtype):
    """The first 16 channels of every token take uniformly random residuals (their
    four lanes per chunk hold 1.3-2.8 KB, mostly escapes), the others residuals of
    at most 2: chunks of 12-22 KB whose long lanes span several 1-KB staging
    pieces.  GPU stream == oracle stream, exact decode."""
    L, KV, H, T, D, K = 2, 2, 2, 700, 128, 1024
    n = L * KV * H * T * D
    rng = np.random.default_rng(7 + dtype)
    hi, dt = (256, np.uint8) if dtype == synth.FP8 else (1 << 16, np.uint16)
    t = rng.integers(0, hi, n)
    p = np.clip(t + rng.integers(-2, 3, n), 0, hi - 1)
    hot = (np.arange(n) % D) < 16
    p[hot] = rng.integers(0, hi, int(hot.sum()))
    tn, pn = t.astype(dt), p.astype(dt)
    po = oracle.kv_params(dtype, L, KV, H, D, T, K, 256)
    bins, _, _ = oracle.calibrate(po, tn, pn)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    lens = np.diff(offs.astype(np.int64))
    assert lens.max() > 1024 and np.diff(offs[::32].astype(np.int64)).max() <= 32768   # the shape meant
    tdt = torch.uint8 if dtype == synth.FP8 else torch.int16
    td = torch.from_numpy(tn.view(np.int16) if dtype == synth.BF16 else tn).to(tdt).cuda()
    pd = torch.from_numpy(pn.view(np.int16) if dtype == synth.BF16 else pn).to(tdt).cuda()
    codec = nat.Codec(nat.kv_params(dtype, L, KV, H, D, T, K, 256))
    codec.calibrate(td, pd)
    codec.build_tables()
    total = codec.encode(td, pd)
    assert codec.check() == nat.SKV_OK and total == bs.size
    assert np.array_equal(codec.bitstream[:total].cpu().numpy(), bs)
    assert np.array_equal(codec.lane_offsets.cpu().numpy().astype(np.uint64), offs)
    out = torch.empty_like(td)
    codec.decode(pd, out)
    assert codec.check() == nat.SKV_OK and torch.equal(out, td)


@pytest.mark.parametrize("dtype", [synth.FP8, synth.BF16])
@pytest.mark.parametrize("kind", ["uniform", "nan", "signflip", "extremes", "mixture"])
def test_adversarial_bit_exact(nat, dtype, kind):
    """escape-heavy and special-value inputs: GPU stream == oracle stream, exact decode"""
    L, KV, H, T, D = 2, 2, 2, 700, 128
    K = 256 if dtype == synth.FP8 else 128
    n = L * KV * H * T * D
    tn, pn = _adversarial(kind, dtype, n, seed=hash(kind) % 1000 + dtype)
    po = oracle.kv_params(dtype, L, KV, H, D, T, K, 256)
    bins, _, _ = oracle.calibrate(po, tn, pn)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    tdt = torch.uint8 if dtype == synth.FP8 else torch.int16
    td = torch.from_numpy(tn.view(np.int16) if dtype == synth.BF16 else tn).to(tdt).cuda()
    pd = torch.from_numpy(pn.view(np.int16) if dtype == synth.BF16 else pn).to(tdt).cuda()
    codec = nat.Codec(nat.kv_params(dtype, L, KV, H, D, T, K, 256))
    codec.calibrate(td, pd)
    codec.build_tables()
    total = codec.encode(td, pd)
    assert codec.check() == nat.SKV_OK
    assert np.array_equal(codec.bins[: bins.size].cpu().numpy(), bins)
    assert total == bs.size
    assert np.array_equal(codec.bitstream[:total].cpu().numpy(), bs)
    assert np.array_equal(codec.lane_offsets.cpu().numpy().astype(np.uint64), offs)
    out = torch.empty_like(td)
    codec.decode(pd, out)
    assert codec.check() == nat.SKV_OK and torch.equal(out, td)
