"""pipeline.HostPipeline: a KV cache in pinned host memory coded in layer groups
with the host transfers overlapped.  The joined stream and offsets must equal one
whole-cache call byte for byte, and the decoded cache must equal the target."""
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


CASES = [("qwen3-0.6b-1k-fp8", dict(n_layers=5, n_tokens=1024), 2),
         ("qwen3-0.6b-1k-fp8", dict(n_layers=3, n_tokens=700, lane_syms=256), 1),
         ("qwen3-0.6b-8k-bf16", dict(n_layers=3, n_heads=4, n_tokens=1100, lane_syms=512), 2)]


@pytest.mark.parametrize("name,kw,group", CASES)
def test_pipeline_matches_one_call(nat, name, kw, group):
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
    out = torch.zeros_like(t)
    pipe = pipeline.HostPipeline(nat.params_for(w), group_layers=group)
    assert len(pipe.groups) == -(-w.n_layers // group)
    for _ in range(2):   # the second run reuses every buffer
        n = pipe.run(h_t, h_p, h_bs, h_off, decode_into=out)
        torch.cuda.synchronize()
        assert pipe.check() == nat.SKV_OK
        assert n == total
        assert torch.equal(h_bs[:n], codec.bitstream[:n].cpu())
        assert np.array_equal(pipe.joined_offsets(h_off.numpy()), codec.lane_offsets.cpu().numpy().view(np.uint64))
        assert torch.equal(out, t)
        out.zero_()
