"""The exponent residual model (SKV_MODEL_EXPONENT, FP8) on the GPU against the
oracle: base bins and sums from calibration, the bitstream and lane offsets
byte for byte, and the decoded cache; dense and paged pools; planted escapes;
the whole 1K-token Qwen3-0.6B-shaped cache."""
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


def _oracle(w, tn, pn):
    po = oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                          w.n_calib, model=1)
    bins, sums, _ = oracle.calibrate(po, tn, pn)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    return bins, sums, bs, offs


def _check(nat, w, t, p):
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    bins, sums, bs, offs = _oracle(w, tn, pn)
    td, pd = t.cuda(), p.cuda()
    codec = nat.Codec(nat.params_for(w, model=nat.SKV_MODEL_EXPONENT))
    s_d = torch.zeros(bins.size, dtype=torch.int32, device="cuda")
    codec.calibrate(td, pd, sum_abs=s_d)
    codec.build_tables()
    total = codec.encode(td, pd)
    assert codec.check() == nat.SKV_OK
    assert np.array_equal(codec.bins[:bins.size].cpu().numpy(), bins)
    assert np.array_equal(s_d.cpu().numpy().view(np.uint32), sums)
    assert total == bs.size and np.array_equal(codec.bitstream[:total].cpu().numpy(), bs)
    assert np.array_equal(codec.lane_offsets.cpu().numpy().view(np.uint64), offs)
    out = torch.zeros_like(td)
    codec.decode(pd, out)
    assert codec.check() == nat.SKV_OK and torch.equal(out, td)
    return codec, total


SMALL = [dict(n_layers=1, n_tokens=300, lane_syms=64, n_heads=2),
         dict(n_layers=2, n_tokens=777, lane_syms=256, n_heads=3),
         dict(n_layers=1, n_tokens=1024, lane_syms=1024, n_heads=8, head_dim=64),
         dict(n_layers=1, n_tokens=100, lane_syms=16, n_heads=1, head_dim=16)]


@pytest.mark.parametrize("kw", SMALL)
def test_model_exponent_bit_exact(nat, kw):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(**kw)
    t, p = synth.gen_kv(w, "cpu")
    _check(nat, w, t, p)


def test_model_exponent_escapes(nat):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_tokens=512, lane_syms=128, n_heads=2)
    t, p = synth.gen_kv(w, "cpu")
    tf = t.reshape(-1).clone()
    g = torch.Generator().manual_seed(11)
    idx = torch.randperm(tf.numel(), generator=g)[:500]
    tf[idx] = (p.reshape(-1)[idx].to(torch.int64) + 128 + torch.randint(0, 100, (500,), generator=g)).to(torch.uint8)
    _check(nat, w, tf.reshape(t.shape), p)


def test_model_exponent_paged(nat):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=2, n_tokens=1000, n_heads=4)
    t, p = synth.gen_kv(w, "cuda")
    codec = nat.Codec(nat.params_for(w, model=nat.SKV_MODEL_EXPONENT))
    codec.calibrate(t, p)
    codec.build_tables()
    total = codec.encode(t, p)
    tp, pp, table, n_blocks = synth.to_paged(t, p, 16, seed=3)
    lay = nat.paged_layout(table, n_blocks, 16)
    prm = nat.params_for(w, model=nat.SKV_MODEL_EXPONENT)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    bins = torch.empty_like(codec.bins)
    assert nat.skv_calibrate_paged(prm, lay, tp, pp, bins, status) == nat.SKV_OK
    assert torch.equal(bins, codec.bins)
    bs = torch.empty_like(codec.bitstream)
    off = torch.empty_like(codec.lane_offsets)
    st, n = nat.skv_encode_paged(prm, lay, tp, pp, codec.tables, bins, bs, codec.cap, off, codec.workspace,
                                 codec.workspace.numel(), status)
    assert st == nat.SKV_OK and n == total and torch.equal(bs[:n], codec.bitstream[:n])
    out = torch.zeros_like(tp)
    assert nat.skv_decode_paged(prm, lay, bs, n, off, pp, codec.tables, bins, out, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK and torch.equal(out, tp)


def test_model_exponent_full_1k(nat):
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"]
    t, p = synth.gen_kv(w, "cpu")
    codec, total = _check(nat, w, t, p)
    # and it codes the cache smaller than the per-channel model
    c0 = nat.Codec(nat.params_for(w))
    td, pd = t.cuda(), p.cuda()
    c0.calibrate(td, pd)
    c0.build_tables()
    assert total < 0.92 * c0.encode(td, pd)
