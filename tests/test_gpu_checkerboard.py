"""Checkerboard context on the GPU (skv_ctx_means) against the oracle: the
odd rows' shifted means bit for bit (small and full-width maps, ragged tiles,
extreme values, weights outside [-8, 8]), every row of the full 32K-token
stream, and the two-pass round trip through the COEF calls with streams equal
to the oracle's."""
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


def _gpu_ctx(nat, V, U, s1, s2, qe, mo):
    Vd, Ud = torch.as_tensor(V).cuda(), torch.as_tensor(U).cuda()
    qd, md = torch.as_tensor(qe).cuda(), torch.as_tensor(mo).cuda()
    out = torch.full_like(md, float("nan"))
    nb = nat.skv_ctx_scratch_bytes(mo.shape[0], qe.shape[1], V.shape[0])
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    status = torch.ones(4, dtype=torch.int32, device="cuda")
    st = nat.skv_ctx_means(nat.ctx_map(Vd, Ud, s1, s2), qd, qe.shape[0], md, mo.shape[0], qe.shape[1], out, scratch,
                           status)
    assert st == nat.SKV_OK
    torch.cuda.synchronize()
    assert nat.skv_read_status(status) == nat.SKV_OK
    return out.cpu().numpy()


@pytest.mark.parametrize("C,R,n_e,n_o", [(256, 64, 33, 33), (96, 32, 5, 4), (2048, 1024, 300, 300), (512, 1024, 131, 130),
                                        (416, 160, 258, 257)])
def test_ctx_means_match_oracle(nat, C, R, n_e, n_o):
    rng = np.random.default_rng(C + R + n_o)
    V = rng.integers(-8, 9, (R, C)).astype(np.int8)
    U = rng.integers(-8, 9, (C, R)).astype(np.int8)
    V[0, :3] = [127, -128, 9]
    U[1, :2] = [-100, 50]
    qe = rng.integers(-300, 301, (n_e, C)).astype(np.int16)
    qe[0, :4] = [32767, -32768, 127, -128]
    mo = (rng.standard_normal((n_o, C)) * 50).astype(np.float32)
    mo[0, :3] = [1e9, -3.97, 0.03125]
    for s1, s2 in [(6, 8), (0, 3)]:
        want = oracle.ctx_means(V, U, s1, s2, qe, mo)
        got = _gpu_ctx(nat, V, U, s1, s2, qe, mo)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def _coef_gpu(nat, w, q, mu, beta):
    p = nat.coef_params(q.shape[0], q.shape[1], w.lane_syms)
    codec = nat.Codec(p)
    codec.calibrate(None, beta)
    codec.build_tables()
    n = codec.encode(q, mu)
    assert codec.check() == nat.SKV_OK
    return codec, n


def test_two_pass_round_trip(nat):
    w = synth.WORKLOADS["hybrid-coef-32k-x2048"].scaled(n_tokens=257, lane_syms=128)
    qe, qo, me, mo, beta, V, U = synth.gen_coef_checkerboard(w, "cuda")
    s1, s2 = synth.CTX_SHIFT1, synth.CTX_SHIFT2
    C = qe.shape[1]
    scratch = torch.empty(nat.skv_ctx_scratch_bytes(qo.shape[0], C, V.shape[0]), dtype=torch.uint8, device="cuda")
    cmap = nat.ctx_map(V, U, s1, s2)
    status = torch.ones(4, dtype=torch.int32, device="cuda")
    mo2 = torch.empty_like(mo)
    assert nat.skv_ctx_means(cmap, qe, qe.shape[0], mo, qo.shape[0], C, mo2, scratch, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    ce, ne = _coef_gpu(nat, w, qe, me, beta)
    co, no = _coef_gpu(nat, w, qo, mo2, beta)
    # the streams equal the oracle's
    on = lambda x: x.cpu().numpy()
    mo2_o = oracle.ctx_means(on(V), on(U), s1, s2, on(qe), on(mo))
    assert np.array_equal(on(mo2).view(np.uint32), mo2_o.view(np.uint32))
    for q, mu, codec, n in [(qe, me, ce, ne), (qo, mo2, co, no)]:
        po = oracle.coef_params(q.shape[0], C, w.lane_syms)
        bins, _, _ = oracle.calibrate(po, None, on(beta))
        fr, cum = oracle.build_tables(po)
        st, bs, offs = oracle.encode(po, fr, cum, bins, on(q).reshape(-1), on(mu).reshape(-1))
        assert st == oracle.OK and n == bs.size and np.array_equal(on(codec.bitstream[:n]), bs)
    # decode: even rows, context from them, odd rows
    qe_d = torch.zeros_like(qe)
    ce.decode(me, qe_d)
    assert ce.check() == nat.SKV_OK and torch.equal(qe_d, qe)
    mo3 = torch.empty_like(mo)
    assert nat.skv_ctx_means(cmap, qe_d, qe.shape[0], mo, qo.shape[0], C, mo3, scratch, status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    qo_d = torch.zeros_like(qo)
    co.decode(mo3, qo_d)
    assert co.check() == nat.SKV_OK and torch.equal(qo_d, qo)


def test_full_size_every_row(nat):
    """the full 32K-token stream's context (16384 odd rows, rank 1024): every odd
    row's shifted means against the oracle (row blocks in host threads)"""
    import concurrent.futures as cf
    import os
    w = synth.WORKLOADS["hybrid-coef-32k-x2048"]
    qe, qo, me, mo, beta, V, U = synth.gen_coef_checkerboard(w, "cuda")
    s1, s2 = synth.CTX_SHIFT1, synth.CTX_SHIFT2
    C, n_e, n_o = qe.shape[1], qe.shape[0], qo.shape[0]
    scratch = torch.empty(nat.skv_ctx_scratch_bytes(n_o, C, V.shape[0]), dtype=torch.uint8, device="cuda")
    mo2 = torch.empty_like(mo)
    status = torch.ones(4, dtype=torch.int32, device="cuda")
    assert nat.skv_ctx_means(nat.ctx_map(V, U, s1, s2), qe, n_e, mo, n_o, C, mo2, scratch,
                             status) == nat.SKV_OK
    assert nat.skv_read_status(status) == nat.SKV_OK
    Vh, Uh, qh, mh = V.cpu().numpy(), U.cpu().numpy(), qe.cpu().numpy(), mo.cpu().numpy()
    got = mo2.cpu().numpy().view(np.uint32)
    step = 256

    def block(t0):
        t1 = min(t0 + step, n_o)
        want = oracle.ctx_means(Vh, Uh, s1, s2, qh[t0:min(t1 + 1, n_e)], mh[t0:t1])
        return t0 if not np.array_equal(got[t0:t1], want.view(np.uint32)) else None

    with cf.ThreadPoolExecutor(os.cpu_count() or 4) as ex:
        bad = [t for t in ex.map(block, range(0, n_o, step)) if t is not None]
    assert not bad, f"row blocks {bad[:5]} differ"


def test_ctx_rejects_bad_shapes(nat):
    V = torch.zeros((64, 100), dtype=torch.int8, device="cuda")
    U = torch.zeros((100, 64), dtype=torch.int8, device="cuda")
    z = torch.zeros(4096, dtype=torch.float32, device="cuda")
    st = nat.skv_ctx_means(nat.ctx_map(V, U, 6, 8), z, 2, z, 2, 100, z, z, z)   # n_coef not a multiple of 32
    assert st == nat.SKV_ERR_INVALID_ARG
    st = nat.skv_ctx_means(nat.ctx_map(V[:, :96], U[:96], 6, 8), z, 1, z, 2, 96, z, z, z)   # more odd than even rows
    assert st == nat.SKV_ERR_INVALID_ARG


def test_ctx_wait_gives_up_without_hanging(nat):
    """a tensor-core tile whose operands never arrive: its MMA thread stops waiting
    after about a second, the call reports a timeout, and the context stays usable"""
    import time
    scratch = torch.zeros(48 * 1024 // 4, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    assert nat.skv_selftest_ctx_wait(scratch, status) == nat.SKV_OK
    st = nat.skv_read_status(status)
    dt = time.perf_counter() - t0
    assert st == nat.SKV_ERR_TIMEOUT and dt < 10.0
    rng = np.random.default_rng(3)
    V = rng.integers(-8, 9, (64, 96)).astype(np.int8)
    U = rng.integers(-8, 9, (96, 64)).astype(np.int8)
    qe = rng.integers(-300, 301, (9, 96)).astype(np.int16)
    mo = (rng.standard_normal((8, 96)) * 50).astype(np.float32)
    want = oracle.ctx_means(V, U, 6, 8, qe, mo)
    assert np.array_equal(_gpu_ctx(nat, V, U, 6, 8, qe, mo).view(np.uint32), want.view(np.uint32))
