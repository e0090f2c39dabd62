"""Paged pools (skv_*_paged): the same bins, bitstream and lane offsets as the
dense calls on the gathered cache, and a decode that writes exactly the target
rows of the pool.  Ragged last blocks, several block sizes, FP8 and BF16, and an
out-of-range block-table entry (flagged, its rows never written)."""
import numpy as np
import pytest
import torch

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


CASES = [("qwen3-0.6b-1k-fp8", dict(n_layers=2, n_tokens=1000), 16),
         ("qwen3-0.6b-1k-fp8", dict(n_layers=1, n_heads=3, n_tokens=777, lane_syms=256), 1),
         ("qwen3-0.6b-1k-fp8", dict(n_layers=2, n_tokens=1024), 256),
         ("qwen3-0.6b-8k-bf16", dict(n_layers=2, n_heads=4, n_tokens=900, lane_syms=512), 32)]


def _dense(nat, w, t, p):
    codec = nat.Codec(nat.params_for(w))
    sums = torch.zeros(codec.sz["channels"], dtype=torch.int32, device="cuda")
    codec.calibrate(t, p, sum_abs=sums)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    return codec, sums, total


@pytest.mark.parametrize("name,kw,B", CASES)
def test_paged_equals_dense(nat, name, kw, B):
    w = synth.WORKLOADS[name].scaled(**kw)
    t, p, _ = synth.gen_workload(w, "cuda")
    codec, sums, total = _dense(nat, w, t, p)
    tp, pp, table, n_blocks = synth.to_paged(t, p, B, seed=B)
    lay = nat.paged_layout(table, n_blocks, B)
    prm = nat.params_for(w)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    bins = torch.empty_like(codec.bins)
    sums2 = torch.zeros_like(sums)
    assert nat.skv_calibrate_paged(prm, lay, tp, pp, bins, status, sum_abs=sums2) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    nch = codec.sz["channels"]
    assert torch.equal(bins[:nch], codec.bins[:nch]) and torch.equal(sums2, sums)
    bs = torch.full_like(codec.bitstream, 0xAB)
    off = torch.full_like(codec.lane_offsets, -1)
    st, n = nat.skv_encode_paged(prm, lay, tp, pp, codec.tables, bins, bs, codec.cap, off, codec.workspace,
                                 codec.workspace.numel(), status)
    assert st == nat.SKV_OK and nat.skv_read_status(status) == nat.SKV_OK
    assert n == total and torch.equal(bs[:n], codec.bitstream[:n]) and torch.equal(off, codec.lane_offsets)
    out = torch.zeros_like(tp)
    assert nat.skv_decode_paged(prm, lay, bs, n, off, pp, codec.tables, bins, out, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    # the target rows hold the target; unused blocks and rows past the last token stay zero
    assert torch.equal(out, tp)


def test_paged_matches_oracle(nat, orc):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_heads=2, n_tokens=600, lane_syms=128)
    t, p, _ = synth.gen_workload(w, "cpu")
    op = orc.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib)
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    obins, _, _ = orc.calibrate(op, tn, pn)
    fr, cum = orc.build_tables(op)
    ost, obs, ooff = orc.encode(op, fr, cum, obins, tn, pn)
    assert ost == orc.OK
    tp, pp, table, n_blocks = synth.to_paged(t.cuda(), p.cuda(), 64, seed=5)
    lay = nat.paged_layout(table, n_blocks, 64)
    prm = nat.params_for(w)
    sz = nat.sizes(prm)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    bins = torch.empty(max(sz["channels"], 16), dtype=torch.uint8, device="cuda")
    tables = torch.empty(sz["tables_bytes"], dtype=torch.uint8, device="cuda")
    assert nat.skv_calibrate_paged(prm, lay, tp, pp, bins, status) == nat.SKV_OK
    assert nat.skv_build_tables(prm, tables) == nat.SKV_OK
    bs = torch.empty(sz["max_bitstream"], dtype=torch.uint8, device="cuda")
    off = torch.empty(sz["lanes"] + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(sz["workspace"], 256), dtype=torch.uint8, device="cuda")
    st, n = nat.skv_encode_paged(prm, lay, tp, pp, tables, bins, bs, bs.numel(), off, ws, ws.numel(), status)
    assert st == nat.SKV_OK
    assert np.array_equal(bins[:sz["channels"]].cpu().numpy(), obins)
    assert n == obs.size and np.array_equal(bs[:n].cpu().numpy(), obs)
    assert np.array_equal(off.cpu().numpy().view(np.uint64), ooff)


def test_paged_bad_block_entry_is_flagged(nat):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_heads=2, n_tokens=512, lane_syms=256)
    t, p, _ = synth.gen_workload(w, "cuda")
    codec, _, total = _dense(nat, w, t, p)
    tp, pp, table, n_blocks = synth.to_paged(t, p, 32, spare_blocks=1, seed=9)
    spare = sorted(set(range(n_blocks)) - set(table.tolist()))[0]
    prm = nat.params_for(w)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    # decode with one entry pointing past the pool: flagged, and no row outside
    # the listed blocks is written (the spare block stays zero)
    bad = table.clone()
    bad[3] = n_blocks + 5
    lay_bad = nat.paged_layout(bad, n_blocks, 32)
    out = torch.zeros_like(tp)
    st = nat.skv_decode_paged(prm, lay_bad, codec.bitstream, total, codec.lane_offsets, pp, codec.tables,
                              codec.bins, out, status)
    assert st == nat.SKV_OK and nat.skv_read_status(status) == nat.SKV_ERR_INVALID_ARG
    assert int(out[:, :, spare].abs().sum()) == 0
    # encode with it: flagged too
    bs = torch.empty_like(codec.bitstream)
    off = torch.empty_like(codec.lane_offsets)
    st, _ = nat.skv_encode_paged(prm, lay_bad, tp, pp, codec.tables, codec.bins, bs, codec.cap, off,
                                 codec.workspace, codec.workspace.numel(), status)
    assert st == nat.SKV_OK and nat.skv_read_status(status) == nat.SKV_ERR_INVALID_ARG


def test_paged_full_size_equals_dense(nat):
    """the 128K Qwen3-32B-shaped cache in 16-token pages: bins, stream and offsets
    equal the dense call's (itself checked chunk by chunk against the oracle) and
    decoding into the pool restores every target row"""
    w = synth.WORKLOADS["qwen3-32b-128k-fp8"]
    free, _ = torch.cuda.mem_get_info()
    if free < 8 * w.raw_bytes:
        pytest.skip(f"needs {8 * w.raw_bytes / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")
    t, p, _ = synth.gen_workload(w, "cuda")
    prm = nat.params_for(w)
    codec = nat.Codec(prm, bitstream_capacity=w.raw_bytes)
    codec.calibrate(t, p)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    tp, pp, table, n_blocks = synth.to_paged(t, p, 16, seed=16)
    del t, p
    torch.cuda.empty_cache()
    lay = nat.paged_layout(table, n_blocks, 16)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    bins = torch.empty_like(codec.bins)
    assert nat.skv_calibrate_paged(prm, lay, tp, pp, bins, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    nch = codec.sz["channels"]
    assert torch.equal(bins[:nch], codec.bins[:nch])
    bs = torch.full_like(codec.bitstream, 0xAB)
    off = torch.full_like(codec.lane_offsets, -1)
    st, n = nat.skv_encode_paged(prm, lay, tp, pp, codec.tables, bins, bs, codec.cap, off, codec.workspace,
                                 codec.workspace.numel(), status)
    assert st == nat.SKV_OK and nat.skv_read_status(status) == nat.SKV_OK
    assert n == total and torch.equal(bs[:n], codec.bitstream[:n]) and torch.equal(off, codec.lane_offsets)
    out = torch.zeros_like(tp)
    assert nat.skv_decode_paged(prm, lay, bs, n, off, pp, codec.tables, bins, out, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    assert torch.equal(out, tp)
