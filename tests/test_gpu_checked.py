"""The checked build (libskv_checked.so, -DSKV_CHECKED=1) on the small parity,
ragged-shape, adversarial and corrupt-stream cases: every shared-memory access,
table / word-buffer / scratch-slot cursor, decoder output row and stream copy
is checked inside the kernels (a failed check is counted and skipped, never a
trap), the results still equal the oracle's, and no check may fail.  This
stands in for a memory checker, which this environment does not offer."""
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
    from lossless_kv_cache_fp8_gb300 import build, native
    path = build.build(checked=True)
    native.use_library(path)
    st, n, site = native.skv_checked_failures()   # start from a clean record
    assert st == native.SKV_OK
    yield native
    native.use_library(None)


def _no_failures(nat):
    st, n, site = nat.skv_checked_failures()
    assert st == nat.SKV_OK
    assert n == 0, f"{n} failed checks, first at site {site}"


def test_ordinary_build_has_no_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from lossless_kv_cache_fp8_gb300 import build, native
    L = native.load(build.LIB)
    import ctypes as C
    n, s = C.c_uint32(0), C.c_uint32(0)
    assert L.skv_checked_failures(C.byref(n), C.byref(s)) == native.SKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("i", range(10))
def test_checked_small_bit_exact(nat, i):
    from test_gpu_parity import SMALL, full_compare
    full_compare(nat, SMALL[i])
    _no_failures(nat)


@pytest.mark.parametrize("dtype", [synth.FP8, synth.BF16])
@pytest.mark.parametrize("kind", ["uniform", "nan", "extremes", "mixture"])
def test_checked_adversarial(nat, dtype, kind):
    from test_gpu_parity import test_adversarial_bit_exact
    test_adversarial_bit_exact(nat, dtype, kind)
    _no_failures(nat)


def test_checked_corrupt_streams_and_models(nat):
    from test_gpu_parity import test_corrupt_streams_reported
    test_corrupt_streams_reported(nat)
    _no_failures(nat)
    # exponent residual model and paged pools on a small ragged cache
    w = synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=2, n_heads=3, n_tokens=777, lane_syms=256)
    t, p = synth.gen_kv(w, "cpu")
    tn, pn = t.numpy().reshape(-1), p.numpy().reshape(-1)
    po = oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms,
                          w.n_calib, model=1)
    bins, _, _ = oracle.calibrate(po, tn, pn)
    fr, cum = oracle.build_tables(po)
    st, bs, offs = oracle.encode(po, fr, cum, bins, tn, pn)
    assert st == oracle.OK
    codec = nat.Codec(nat.params_for(w, model=nat.SKV_MODEL_EXPONENT))
    td, pd = t.cuda(), p.cuda()
    codec.calibrate(td, pd)
    codec.build_tables()
    total = codec.encode(td, pd)
    assert codec.check() == nat.SKV_OK and total == bs.size
    assert np.array_equal(codec.bitstream[:total].cpu().numpy(), bs)
    out = torch.zeros_like(td)
    codec.decode(pd, out)
    assert codec.check() == nat.SKV_OK and torch.equal(out, td)
    _no_failures(nat)


def test_checked_both_chunk_copies(nat):
    """many short chunks per warp (16-position lanes): early chunks are placed by
    the lane-by-lane copy, the last wave through the staging slots; no check fails
    and the stream equals the oracle's"""
    from test_gpu_parity import full_compare
    full_compare(nat, synth.WORKLOADS["qwen3-0.6b-1k-fp8"].scaled(n_layers=4, lane_syms=16))
    _no_failures(nat)
