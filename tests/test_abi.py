"""CPU checks of the C ABI library: it builds, loads, exports every function
include/srh.h declares, and its host-side guards behave as the pages state.
No kernel runs here (these tests need no GPU)."""
import ctypes
import shutil

import pytest

from oracle import srh_oracle as O

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc not available")


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_retrieval_host_gb300 import abi as a
    return a


def test_library_exports_every_header_function(abi):
    lib = abi.load()
    names = abi.header_functions()
    for must in ("fm_score", "fm_select", "kvswap_stage", "lsa_attend", "srh_create", "srh_destroy",
                 "srh_get_stats", "srh_check_error", "srh_error_string"):
        assert must in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(n for n, _, _ in abi.SIGNATURES) == sorted(names)


def test_error_strings(abi):
    for code in range(0, -8, -1):
        s = abi.error_string(code)
        assert s and s != "unknown error"
    assert abi.error_string(-99) == "unknown error"
    assert "stored" in abi.error_string(abi.SRH_ERR_NOT_STORED)


def test_pinned_required_bytes_matches_formula(abi):
    ratios = [4] * 20 + [128] * 21
    for ctx_len in (8192, 262144, 1048576, 64, 65):
        for batch in (1, 3):
            cfg = abi.make_config(batch=batch, layer_ratios=ratios, gpu_chunks=512, index_topk=512,
                                  context_len=ctx_len)
            assert abi.srh_pinned_required_bytes(cfg) == batch * O.required_pinned_bytes(ctx_len, ratios)


def test_gpu_chunks_below_topk_is_rejected(abi):
    """Section 故障排查, error 2."""
    cfg = abi.make_config(batch=1, layer_ratios=[4], gpu_chunks=256, index_topk=512, context_len=8192)
    with pytest.raises(abi.SrhError) as ei:
        abi.srh_create(cfg)
    assert ei.value.code == abi.SRH_ERR_INVALID
    assert "GPU_CHUNKS must be >= index_topk" in str(ei.value)
    with pytest.raises(abi.SrhError) as ei:
        abi.srh_pinned_required_bytes(cfg)
    assert ei.value.code == abi.SRH_ERR_INVALID


def test_pinned_cap_exceeded_reports_required_and_cap(abi):
    """Section 故障排查, error 3; the 8K example log's pinned_mib=84 (21 ratio-4 layers)."""
    cfg = abi.make_config(batch=1, layer_ratios=[4] * 21, gpu_chunks=512, index_topk=512,
                          context_len=8192, pinned_cap_bytes=64 << 20)
    with pytest.raises(abi.SrhError) as ei:
        abi.srh_create(cfg)
    assert ei.value.code == abi.SRH_ERR_PINNED_CAP
    assert "required_mib=84 cap_mib=64" in str(ei.value)


@pytest.mark.parametrize("kw", [dict(layer_ratios=[6]), dict(layer_ratios=[2]), dict(gpu_chunks=0),
                                dict(index_topk=0), dict(context_len=0), dict(max_select=100),
                                dict(max_select=5000), dict(gpu_chunks=8192)])
def test_bad_configs_are_invalid(abi, kw):
    base = dict(batch=1, layer_ratios=[4, 128], gpu_chunks=512, index_topk=512, context_len=8192)
    base.update(kw)
    cfg = abi.make_config(**base)
    with pytest.raises(abi.SrhError) as ei:
        abi.srh_create(cfg)
    assert ei.value.code == abi.SRH_ERR_INVALID


def test_bad_kv_dim_is_invalid(abi):
    cfg = abi.make_config(batch=1, layer_ratios=[4], gpu_chunks=512, index_topk=512, context_len=8192)
    cfg.kv_dim = 256
    with pytest.raises(abi.SrhError):
        abi.srh_create(cfg)


def test_null_context_calls_are_invalid(abi):
    lib = abi.load()
    assert lib.srh_check_error(None) == abi.SRH_ERR_INVALID
    assert lib.srh_selftest_wait_timeout(None, 1000, None) == abi.SRH_ERR_INVALID
    assert lib.fm_score(None, None, 1, None, ctypes.c_float(1.0), None, 0, None, None) == abi.SRH_ERR_INVALID
    assert lib.lsa_attend(None, -1, None, 64, None, None, None, None, None, None) == abi.SRH_ERR_INVALID
    lib.srh_destroy(None)


def test_null_host_loop_calls_are_invalid(abi):
    """The native host loop's entry points refuse a missing context or loop
    before any GPU call, and its destroy accepts NULL."""
    lib = abi.load()
    out = ctypes.c_void_p(12345)
    bias = (ctypes.c_float * 3)(0.0, 0.0, 0.0)
    rc = lib.srh_hostloop_create(None, None, 1, None, None, None, None, None, 64, ctypes.c_float(1.0), bias, 0, 0,
                                 1, ctypes.c_float(0.5), 0, None, None, None, None, None, None, ctypes.byref(out))
    assert rc == abi.SRH_ERR_INVALID
    assert lib.srh_hostloop_create(None, None, 1, None, None, None, None, None, 64, ctypes.c_float(1.0), bias, 0, 0,
                                   1, ctypes.c_float(0.5), 0, None, None, None, None, None, None,
                                   None) == abi.SRH_ERR_INVALID
    assert lib.srh_hostloop_step(None, 0, None, None, None, None, None) == abi.SRH_ERR_INVALID
    assert lib.srh_hostloop_wait(None, 0) == abi.SRH_ERR_INVALID
    assert lib.srh_hostloop_sync(None) == abi.SRH_ERR_INVALID
    lib.srh_hostloop_destroy(None)


def test_every_entry_point_refuses_null_arguments(abi):
    """Every int-returning export, called with every pointer NULL and every
    number zero, returns SRH_ERR_INVALID before any GPU call; the pointer
    getter returns NULL and the destroy calls accept NULL (the header's error
    behaviour, checked for each function the binding declares)."""
    lib = abi.load()
    numbers = (ctypes.c_int, ctypes.c_long, ctypes.c_longlong, ctypes.c_uint, ctypes.c_ulonglong, ctypes.c_size_t)
    checked = []
    for name, res, argtypes in abi.SIGNATURES:
        args = [0 if t in numbers else 0.0 if t in (ctypes.c_float, ctypes.c_double) else None for t in argtypes]
        r = getattr(lib, name)(*args)
        if res is ctypes.c_int:
            assert r == abi.SRH_ERR_INVALID, (name, r)
            checked.append(name)
        elif isinstance(res, type) and issubclass(res, ctypes._Pointer):
            assert not r, name
    assert len(checked) >= 25 and {"fm_score", "fm_select", "kvswap_stage", "lsa_attend"} <= set(checked)
