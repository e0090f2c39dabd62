"""skv_encode_noalloc: the encode entry point for callers that cannot allocate
device memory (for example code that a host framework hands only its input and
output buffers, or code running after another pool has claimed the device's
memory).  It uses a fixed scratch array inside libskv.so instead of a
caller-provided workspace.

Checked through the C ABI against skv_encode on two calls in a row with
different inputs, so the second call also shows that the first call's leftovers
in the shared scratch do not leak into its output.  This file is collected last
so that a run stopping at the first failure has already run every other test.
"""
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


def _encode_both(nat, w):
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(nat.params_for(w))
    codec.calibrate(t, c)
    codec.build_tables()
    ref_total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    ref_bs = codec.bitstream[:ref_total].clone()
    ref_off = codec.lane_offsets.clone()
    # the same call without a workspace
    bs = torch.full_like(codec.bitstream, 0xAB)
    off = torch.full_like(codec.lane_offsets, -1)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    st, total = nat.skv_encode_noalloc(codec.p, t, p, codec.tables, codec.bins, bs, codec.cap, off, status)
    assert st == nat.SKV_OK, nat.status_string(st)
    assert nat.skv_read_status(status) == nat.SKV_OK
    return ref_total, ref_bs, ref_off, total, bs, off


def test_noalloc_matches_workspace_encode_twice(nat):
    w1 = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_tokens=1024)
    w2 = synth.WORKLOADS["qwen3-0.6b-8k-bf16"].scaled(n_layers=1, n_heads=4, n_tokens=700, lane_syms=256)
    for w in (w1, w2):
        assert nat.sizes(nat.params_for(w))["workspace"] <= 64 << 20
        ref_total, ref_bs, ref_off, total, bs, off = _encode_both(nat, w)
        assert total == ref_total
        assert torch.equal(bs[:total], ref_bs)
        assert torch.equal(off, ref_off)


def test_noalloc_rejects_streams_beyond_its_scratch(nat):
    p = nat.params_for(synth.WORKLOADS["qwen3-0.6b-8k-bf16"])
    assert nat.sizes(p)["workspace"] > 64 << 20
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    st, _ = nat.skv_encode_noalloc(p, dummy, dummy, dummy, dummy, dummy, 16, dummy, status)
    assert st == nat.SKV_ERR_UNSUPPORTED
