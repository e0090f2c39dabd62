"""pipeline.HostPipeline: a KV cache in pinned host memory coded in layer groups
with the host transfers overlapped.  The joined stream and offsets must equal one
whole-cache call byte for byte, and the decoded cache must equal the target."""
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


CASES = [("qwen3-0.6b-1k-fp8", dict(n_layers=5, n_tokens=1024), 2),
         ("qwen3-0.6b-1k-fp8", dict(n_layers=3, n_tokens=700, lane_syms=256), 1),
         ("qwen3-0.6b-8k-bf16", dict(n_layers=3, n_heads=4, n_tokens=1100, lane_syms=512), 2)]


@pytest.mark.parametrize("name,kw,group", CASES)
def test_pipeline_matches_one_call(nat, name, kw, group):
    """skv_encode_host / skv_decode_host through pipeline.HostPipeline"""
    from lossless_kv_cache_fp8_gb300 import pipeline
    w = synth.WORKLOADS[name].scaled(**kw)
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(nat.params_for(w))
    codec.calibrate(t, c)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    h_t = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h_p = torch.empty(p.shape, dtype=p.dtype, pin_memory=True)
    h_t.copy_(t)
    h_p.copy_(p)
    h_bs = torch.full((codec.cap,), 0xAB, dtype=torch.uint8, pin_memory=True)
    h_off = torch.full(codec.lane_offsets.shape, -1, dtype=torch.int64, pin_memory=True)
    h_out = torch.zeros(t.shape, dtype=t.dtype, pin_memory=True)
    pipe = pipeline.HostPipeline(nat.params_for(w), group_layers=group)
    assert len(pipe.groups) == -(-w.n_layers // group)
    for _ in range(2):   # the second run reuses every buffer
        n = pipe.run(h_t, h_p, h_bs, h_off, decode_into=h_out)
        assert pipe.check() == nat.SKV_OK
        assert n == total
        assert torch.equal(h_bs[:n], codec.bitstream[:n].cpu())
        assert torch.equal(h_off, codec.lane_offsets.cpu())
        assert torch.equal(pipe.bins[:codec.bins.numel()], codec.bins)
        assert torch.equal(h_out, t.cpu())
        h_out.zero_()


def test_host_calls_report_capacity_and_corruption(nat):
    """a group buffer smaller than a group's stream gives SKV_ERR_CAPACITY; offsets
    that do not end at n_bytes give SKV_ERR_CORRUPT before anything runs"""
    from lossless_kv_cache_fp8_gb300 import pipeline
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=2, n_tokens=512)
    t, p, _ = synth.gen_workload(w, "cuda")
    h_t = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h_p = torch.empty(p.shape, dtype=p.dtype, pin_memory=True)
    h_t.copy_(t)
    h_p.copy_(p)
    sz = nat.sizes(nat.params_for(w))
    h_bs = torch.zeros(sz["max_bitstream"], dtype=torch.uint8, pin_memory=True)
    h_off = torch.zeros(sz["lanes"] + 1, dtype=torch.int64, pin_memory=True)
    small = pipeline.HostPipeline(nat.params_for(w), group_layers=1, cap_frac=0.01)
    with pytest.raises(nat.SkvError) as e:
        small.encode(h_t, h_p, h_bs, h_off)
    assert e.value.status == nat.SKV_ERR_CAPACITY
    pipe = pipeline.HostPipeline(nat.params_for(w), group_layers=1)
    n = pipe.encode(h_t, h_p, h_bs, h_off)
    h_out = torch.zeros(t.shape, dtype=t.dtype, pin_memory=True)
    with pytest.raises(nat.SkvError) as e:
        pipe.decode(h_bs, n - 2, h_off, h_p, h_out)
    assert e.value.status == nat.SKV_ERR_CORRUPT
    pipe.decode(h_bs, n, h_off, h_p, h_out)
    assert torch.equal(h_out, t.cpu())


def test_pipeline_exponent_model_in_huge_page_buffers(nat):
    """the exponent residual model through the host calls, with the host buffers
    from pipeline.pinned_empty (huge-page backed, registered): equal to one call"""
    from lossless_kv_cache_fp8_gb300 import pipeline
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=4, n_tokens=600)
    params = nat.params_for(w, model=nat.SKV_MODEL_EXPONENT)
    t, p, c = synth.gen_workload(w, "cuda")
    codec = nat.Codec(params)
    codec.calibrate(t, c)
    codec.build_tables()
    total = codec.encode(t, p)
    assert codec.check() == nat.SKV_OK
    h_t = pipeline.pinned_empty(t.shape, t.dtype)
    h_p = pipeline.pinned_empty(p.shape, p.dtype)
    h_bs = pipeline.pinned_empty((codec.cap,), torch.uint8)
    h_off = pipeline.pinned_empty(tuple(codec.lane_offsets.shape), torch.int64)
    h_out = pipeline.pinned_empty(t.shape, t.dtype)
    assert h_t.is_pinned() and h_out.is_pinned() and h_t.shape == t.shape and h_t.dtype == t.dtype
    h_t.copy_(t)
    h_p.copy_(p)
    pipe = pipeline.HostPipeline(params, group_layers=3)
    n = pipe.run(h_t, h_p, h_bs, h_off, decode_into=h_out)
    assert pipe.check() == nat.SKV_OK and n == total
    assert torch.equal(h_bs[:n], codec.bitstream[:n].cpu())
    assert torch.equal(h_off, codec.lane_offsets.cpu())
    assert torch.equal(h_out, t.cpu())
