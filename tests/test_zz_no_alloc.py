"""skv_encode_noalloc: the encode entry point for callers that cannot allocate
device memory (for example code that a host framework hands only its input and
output buffers, or code running after another pool has claimed the device's
memory).  It uses a fixed scratch array inside libskv.so instead of a
caller-provided workspace.

Checked through the C ABI against skv_encode on two calls in a row with
different inputs (FP8, BF16 and a coefficient stream), so the later calls also
show that earlier leftovers in the shared scratch do not leak into their output;
at the largest stream the scratch holds and one chunk past it.  This file is
collected last so that a run stopping at the first failure has already run every
other test.
"""
import pytest
import torch

from lossless_kv_cache_fp8_gb300 import synth

pytestmark = pytest.mark.gpu
SCRATCH = 64 << 20


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
    codec.calibrate(None if w.dtype == synth.COEF else t, c)
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


def _check_same(nat, w):
    assert nat.sizes(nat.params_for(w))["workspace"] <= SCRATCH
    ref_total, ref_bs, ref_off, total, bs, off = _encode_both(nat, w)
    assert total == ref_total
    assert torch.equal(bs[:total], ref_bs)
    assert torch.equal(off, ref_off)


def test_noalloc_matches_workspace_encode_twice(nat):
    w1 = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=1, n_tokens=1024)
    w2 = synth.WORKLOADS["qwen3-0.6b-8k-bf16"].scaled(n_layers=1, n_heads=4, n_tokens=700, lane_syms=256)
    w3 = synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=96, n_coef=1024, lane_syms=512)
    for w in (w1, w2, w3, w1):
        _check_same(nat, w)


def _limit_workload(nat):
    """the FP8 cache of one slice (1 layer, K only, 1 head) with the most
    tokens whose encode scratch fits the array: found with the size query"""
    base = synth.WORKLOADS["qwen3-0.6b-1k-fp8"]
    chunk_tokens = 32 * base.lane_syms // base.head_dim

    def w_of(n_chunks):
        return base.scaled(n_layers=1, n_kv=1, n_heads=1, n_tokens=n_chunks * chunk_tokens)

    n = 1
    while nat.sizes(nat.params_for(w_of(n + 1)))["workspace"] <= SCRATCH:
        n += 1
    return w_of(n), w_of(n + 1), n


def test_noalloc_at_its_limit_and_one_chunk_past(nat):
    w_max, w_over, n = _limit_workload(nat)
    assert nat.sizes(nat.params_for(w_max))["chunks"] == n
    _check_same(nat, w_max)
    p = nat.params_for(w_over)
    assert nat.sizes(p)["workspace"] > SCRATCH and nat.sizes(p)["chunks"] == n + 1
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    st, _ = nat.skv_encode_noalloc(p, dummy, dummy, dummy, dummy, dummy, 16, dummy, status)
    assert st == nat.SKV_ERR_UNSUPPORTED


def test_noalloc_rejects_streams_beyond_its_scratch(nat):
    p = nat.params_for(synth.WORKLOADS["qwen3-0.6b-8k-bf16"])
    assert nat.sizes(p)["workspace"] > SCRATCH
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    st, _ = nat.skv_encode_noalloc(p, dummy, dummy, dummy, dummy, dummy, 16, dummy, status)
    assert st == nat.SKV_ERR_UNSUPPORTED
