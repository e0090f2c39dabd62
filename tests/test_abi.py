"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/skv.h declares, and its pure-host calls (parameter
checks, sizes, status strings) agree with the oracle's geometry."""
import ctypes as C

import pytest

import oracle
from lossless_kv_cache_fp8_gb300 import native, synth


@pytest.fixture(scope="module")
def lib():
    from lossless_kv_cache_fp8_gb300 import build
    build.build()
    return native.lib()


def test_exports_every_declared_symbol(lib):
    names = native.header_functions()
    assert "skv_encode" in names and "skv_decode" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        assert native.status_string(code)
    assert native.status_string(99) == "unknown status"


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_sizes_match_oracle_geometry(lib, name):
    w = synth.WORKLOADS[name]
    p = native.params_for(w)
    assert native.skv_check_params(p) == native.SKV_OK
    s = native.sizes(p)
    po = oracle.coef_params(w.n_tokens, w.n_coef, w.lane_syms) if w.dtype == synth.COEF else \
        oracle.kv_params(w.dtype, w.n_layers, w.n_kv, w.n_heads, w.head_dim, w.n_tokens, w.lane_syms, w.n_calib)
    g = oracle.geometry(po)
    assert s["lanes"] == g["n_lanes"] and s["chunks"] == g["n_chunks"]
    assert s["channels"] == g["n_channels"] and s["tables"] == g["n_tables"]
    assert s["positions"] == w.n_positions
    assert s["max_bitstream"] >= 2 * g["n_lanes"] * 2
    slot = native.SKV_TABLE_SLOT_BYTES if w.dtype == synth.COEF else 0
    assert s["tables_bytes"] == s["tables"] * (native.SKV_TABLE_STRIDE + slot)


def test_param_validation(lib):
    ok = native.kv_params(1, 1, 2, 8, 128, 100, 1024)
    assert native.skv_check_params(ok) == native.SKV_OK
    bad = [native.kv_params(1, 1, 2, 8, 120, 100, 1024),    # head_dim not a multiple of 16
           native.kv_params(1, 1, 2, 8, 1024, 100, 1024),   # head_dim does not divide 512
           native.kv_params(1, 1, 2, 8, 128, 100, 1000),    # lane_syms % 16
           native.kv_params(1, 1, 2, 8, 128, 100, 0),
           native.kv_params(7, 1, 2, 8, 128, 100, 1024),
           native.kv_params(1, 1, 2, 8, 128, 100, 1 << 17),
           native.kv_params(1, 1, 2, 8, 128, 100, 1024, n_calib=70000),
           native.coef_params(10, 0, 64)]
    for p in bad:
        assert native.skv_check_params(p) in (native.SKV_ERR_INVALID_ARG, native.SKV_ERR_UNSUPPORTED)
        assert native.sizes(p)["lanes"] == 0
    v = native.kv_params(1, 1, 2, 8, 128, 100, 1024)
    v.version = 2
    assert native.skv_check_params(v) == native.SKV_ERR_INVALID_ARG


def test_null_arguments_rejected_without_gpu(lib):
    p = native.kv_params(1, 1, 2, 8, 128, 100, 1024)
    assert native.skv_calibrate(p, None, None, None, stream=0) == native.SKV_ERR_INVALID_ARG
    assert native.skv_build_tables(p, None, 0, stream=0) == native.SKV_ERR_INVALID_ARG
    st, _ = native.skv_encode(p, None, None, None, None, None, 0, None, None, 0, None, stream=0)
    assert st == native.SKV_ERR_INVALID_ARG
    assert native.skv_read_status(None, stream=0) == native.SKV_ERR_INVALID_ARG


def test_paged_layout_rejected_without_gpu(lib):
    """every malformed paged layout is refused before anything touches the GPU"""
    p = native.kv_params(1, 1, 2, 8, 128, 100, 1024)
    fake = 1 << 20        # never dereferenced: the layout check fails first
    bad = [native.skv_paged_layout(None, 4, 16),          # no block table
           native.skv_paged_layout(fake + 2, 4, 16),      # table not 4-byte aligned
           native.skv_paged_layout(fake, 0, 16),          # no blocks
           native.skv_paged_layout(fake, 4, 0),           # empty blocks
           native.skv_paged_layout(fake, 4, 24)]          # not a power of two
    for lay in bad:
        assert native.skv_calibrate_paged(p, lay, fake, fake, fake, fake, stream=0) == native.SKV_ERR_INVALID_ARG
        st, _ = native.skv_encode_paged(p, lay, fake, fake, fake, fake, fake, 16, fake, fake, 1 << 30, fake,
                                        stream=0)
        assert st == native.SKV_ERR_INVALID_ARG
        assert native.skv_decode_paged(p, lay, fake, 16, fake, fake, fake, fake, fake, fake,
                                       stream=0) == native.SKV_ERR_INVALID_ARG
    c = native.coef_params(4, 16, 8)
    good = native.skv_paged_layout(fake, 4, 16)
    st, _ = native.skv_encode_paged(c, good, fake, fake, fake, fake, fake, 16, fake, fake, 1 << 30, fake, stream=0)
    assert st == native.SKV_ERR_UNSUPPORTED
    # a null status word is refused by the paged calibration before any launch
    assert native.skv_calibrate_paged(p, good, fake, fake, fake, None, stream=0) == native.SKV_ERR_INVALID_ARG


def test_model_field_validated_without_gpu(lib):
    p = native.kv_params(1, 1, 2, 8, 128, 100, 1024, model=native.SKV_MODEL_EXPONENT)
    assert native.skv_check_params(p) == native.SKV_OK
    p.model = 2
    assert native.skv_check_params(p) == native.SKV_ERR_INVALID_ARG
    b = native.kv_params(2, 1, 2, 8, 128, 100, 1024, model=native.SKV_MODEL_EXPONENT)
    assert native.skv_check_params(b) == native.SKV_ERR_UNSUPPORTED
