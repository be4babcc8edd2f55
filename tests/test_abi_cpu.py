"""The C ABI on a machine without a GPU: the library loads, exports every
function include/pkm.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

import sparse_top_lookup_gb300 as pk

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pkm.h")


@pytest.fixture(scope="module")
def L():
    pk.build()
    return pk.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkm_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "pkm_forward" in names and "pkm_create" in names and "pkm_destroy" in names
    for n in names:
        assert hasattr(L, n), n
    assert sorted(pk.EXPORTED) == names


def test_abi_version_and_strerror(L):
    assert pk.pkm_abi_version() == 3
    for code in range(-11, 1):
        assert pk.pkm_strerror(code) != "unknown error code"
    assert pk.pkm_strerror(-100) == "unknown error code"


def cfg(**kw):
    base = dict(d_q=1024, d_v=1024, max_B=16384, max_H=4, max_n_keys=1024, max_k=32,
                q_dtype=pk.PKM_BF16)
    base.update(kw)
    return pk.make_config(**base)


def test_check_args(L):
    c = cfg()
    assert pk.pkm_check_args(c, 16384, 4, 1024, 32) == pk.PKM_OK
    assert pk.pkm_check_args(c, 0, 4, 1024, 32) == pk.PKM_OK
    assert pk.pkm_check_args(c, 16385, 4, 1024, 32) == pk.PKM_ERR_RANGE
    assert pk.pkm_check_args(c, 1, 5, 1024, 32) == pk.PKM_ERR_RANGE
    assert pk.pkm_check_args(c, 1, 4, 16, 32) == pk.PKM_ERR_RANGE       # k > n_keys
    assert pk.pkm_check_args(c, -1, 4, 1024, 32) == pk.PKM_ERR_INVALID
    assert pk.pkm_check_args(c, 1, 4, 1024, 0) == pk.PKM_ERR_INVALID
    assert pk.pkm_check_args(cfg(d_q=1023), 1, 1, 4, 1) == pk.PKM_ERR_INVALID
    assert pk.pkm_check_args(cfg(d_q=1000), 1, 1, 4, 1) == pk.PKM_ERR_UNSUPPORTED  # TMA stride
    # bf16 with 32 < k <= 64: the CUDA-core path, forward only and within its limits
    assert pk.pkm_check_args(cfg(max_k=64), 1, 1, 64, 48) == pk.PKM_OK
    assert pk.pkm_check_args(cfg(max_k=65), 1, 1, 128, 1) == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(max_k=33, with_backward=1), 1, 1, 64, 1) \
        == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(max_k=33, max_n_keys=4097), 1, 1, 64, 1) \
        == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(max_k=33, d_q=8208), 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(max_k=32, with_backward=1), 1, 1, 64, 32) == pk.PKM_OK
    assert pk.pkm_check_args(cfg(max_k=64, q_dtype=pk.PKM_F32, max_n_keys=1024), 1, 1, 64, 64) \
        == pk.PKM_OK
    assert pk.pkm_check_args(cfg(d_v=1001), 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(max_n_keys=46341), 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(key_dtype=pk.PKM_F32), 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    # fp8 e4m3 is a value-table type only; its rows must be whole 16-byte vectors
    assert pk.pkm_check_args(cfg(value_dtype=pk.PKM_FP8_E4M3), 1, 1, 64, 1) == pk.PKM_OK
    assert pk.pkm_check_args(cfg(value_dtype=pk.PKM_FP8_E4M3, d_v=1000), 1, 1, 64, 1) \
        == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(q_dtype=pk.PKM_FP8_E4M3), 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    c2 = cfg()
    c2.value_dtype = 7
    assert pk.pkm_check_args(c2, 1, 1, 64, 1) == pk.PKM_ERR_UNSUPPORTED
    assert L.pkm_check_args(None, 1, 1, 1, 1) == pk.PKM_ERR_INVALID
    # the backward pass is on the bf16 path, with bf16 or fp32 values
    assert pk.pkm_check_args(cfg(with_backward=1), 1, 1, 64, 1) == pk.PKM_OK
    assert pk.pkm_check_args(cfg(with_backward=1, value_dtype=pk.PKM_F32), 1, 1, 64, 1) \
        == pk.PKM_OK
    assert pk.pkm_check_args(cfg(with_backward=1, value_dtype=pk.PKM_FP8_E4M3), 1, 1, 64, 1) \
        == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_check_args(cfg(with_backward=1, q_dtype=pk.PKM_F32), 1, 1, 64, 1) \
        == pk.PKM_ERR_UNSUPPORTED


def test_null_handle_rejected_before_any_cuda_call(L):
    vp = ctypes.c_void_p
    assert L.pkm_forward(None, 16, 16, 16, 1, 1, 1, 1, 16, None, None, None) == pk.PKM_ERR_INVALID
    assert L.pkm_lookup(None, 16, 16, 1, 1, 1, 1, 16, 16, None) == pk.PKM_ERR_INVALID
    assert L.pkm_gather(None, 16, 1, 1, 1, 1, 16, 16, 16, None) == pk.PKM_ERR_INVALID
    assert L.pkm_forward_host_async(None, 16, 16, 16, 1, 1, 1, 1, 16, None, None, None, 16) \
        == pk.PKM_ERR_INVALID
    assert L.pkm_forward_host(None, 16, 16, 16, 1, 1, 1, 1, 16, None, None, None) \
        == pk.PKM_ERR_INVALID
    assert L.pkm_get_status(None, None) == pk.PKM_ERR_INVALID
    assert L.pkm_backward(None, 16, 16, 16, 1, 1, 1, 1, 16, 16, 16, 16, 16, 16, None) \
        == pk.PKM_ERR_INVALID
    assert L.pkm_backward_read(None, 16, 1, 1, 1, 1, 16, 16, 16, 16, 16, None) \
        == pk.PKM_ERR_INVALID
    assert L.pkm_backward_scores(None, 16, 16, 1, 1, 1, 1, 16, 16, 16, 16, 16, None) \
        == pk.PKM_ERR_INVALID
    assert L.pkm_backward_sparse(None, 16, 16, 16, 1, 1, 1, 1, 16, 16, 16, 16, 16, 16, 16, 16,
                                 None) == pk.PKM_ERR_INVALID
    assert L.pkm_backward_read_sparse(None, 16, 1, 1, 1, 1, 16, 16, 16, 16, 16, 16, 16, None) \
        == pk.PKM_ERR_INVALID
    L.pkm_destroy(None)
    assert L.pkm_create(None, None) == pk.PKM_ERR_INVALID
    h = vp()
    assert L.pkm_create(ctypes.byref(h), None) == pk.PKM_ERR_INVALID
    bad = cfg(d_q=3)
    assert L.pkm_create(ctypes.byref(h), ctypes.byref(bad)) == pk.PKM_ERR_INVALID
    assert h.value is None


def test_fp8_quantiser_rejects_bad_arguments_before_any_cuda_call(L):
    Q = L.pkm_quantize_values_fp8
    assert Q(None, pk.PKM_BF16, 4, 16, 16, None) == pk.PKM_ERR_INVALID
    assert Q(16, pk.PKM_BF16, 0, 16, 16, None) == pk.PKM_ERR_INVALID
    assert Q(16, pk.PKM_BF16, 4, 0, 16, None) == pk.PKM_ERR_INVALID
    assert Q(16, pk.PKM_FP8_E4M3, 4, 16, 16, None) == pk.PKM_ERR_UNSUPPORTED
    assert Q(16, pk.PKM_F32, 4, 24, 16, None) == pk.PKM_ERR_UNSUPPORTED
    assert Q(8, pk.PKM_F32, 4, 16, 16, None) == pk.PKM_ERR_ALIGN
    assert pk.fp8_table_bytes(1 << 20, 1024) == (1 << 30) + (1 << 22)


def test_query_net_rejects_bad_arguments_before_any_cuda_call(L):
    Q = L.pkm_query_net
    assert Q(16, 16, -1, 64, 64, 16, 16, 16, None, None) == pk.PKM_ERR_INVALID
    assert Q(16, 16, 4, 0, 64, 16, 16, 16, None, None) == pk.PKM_ERR_INVALID
    assert Q(16, 16, 4, 72, 64, 16, 16, 16, None, None) == pk.PKM_ERR_UNSUPPORTED  # dim % 16
    assert Q(16, 16, 4, 64, 48, 16, 16, 16, None, None) == pk.PKM_ERR_UNSUPPORTED  # F % 32
    assert Q(16, 16, 0, 64, 64, 16, 16, 16, None, None) == pk.PKM_OK               # B == 0
    assert Q(None, 16, 4, 64, 64, 16, 16, 16, None, None) == pk.PKM_ERR_INVALID
    assert Q(8, 16, 4, 64, 64, 16, 16, 16, None, None) == pk.PKM_ERR_ALIGN
    assert L.pkm_bn_fold(None, 16, 16, 16, 1e-5, 4, 16, 16, None) == pk.PKM_ERR_INVALID
    assert L.pkm_bn_fold(16, 16, 16, 16, 1e-5, 0, 16, 16, None) == pk.PKM_ERR_INVALID


def test_query_net_batch_rejects_bad_arguments_before_any_cuda_call(L):
    Q = L.pkm_query_net_batch
    args = lambda x=16, w=16, B=4, dim=64, F=64, eps=1e-5, ws=16, q=16: \
        Q(x, w, B, dim, F, 16, 16, eps, ws, q, None, None, None, None)
    assert args(B=-1) == pk.PKM_ERR_INVALID
    assert args(dim=0) == pk.PKM_ERR_INVALID
    assert args(eps=-1.0) == pk.PKM_ERR_INVALID
    assert args(eps=float("nan")) == pk.PKM_ERR_INVALID
    assert args(dim=72) == pk.PKM_ERR_UNSUPPORTED  # dim % 16
    assert args(F=48) == pk.PKM_ERR_UNSUPPORTED    # F % 32
    assert args(B=0) == pk.PKM_OK
    assert args(x=None) == pk.PKM_ERR_INVALID
    assert args(ws=None) == pk.PKM_ERR_INVALID
    assert args(x=8) == pk.PKM_ERR_ALIGN
    assert args(ws=8) == pk.PKM_ERR_ALIGN
    # workspace: per-32-row-block sums and squares of every feature, then the
    # joined mean and variance, each region 256-byte aligned
    W = L.pkm_query_net_batch_workspace_bytes
    assert W(-1, 64) == 0 and W(4, 0) == 0
    assert W(32, 64) == 2 * 256 + 2 * 256
    assert W(33, 1024) == 2 * (2 * 1024 * 4) + 2 * (1024 * 4)
    assert W(4096, 1024) >= 2 * 128 * 1024 * 4


def test_flat_entry_points_reject_null_handle_before_any_cuda_call(L):
    assert L.pkm_full_keys(None, 16, 1, 16, 16, None) == pk.PKM_ERR_INVALID
    assert L.pkm_flat_lookup(None, 16, 16, 1, 1, 16, 1, 16, 16, None) == pk.PKM_ERR_INVALID


def test_product_path_refuses_without_library(monkeypatch, tmp_path):
    # No CPU fallback: a missing libpkm.so is an import-time error.
    monkeypatch.setattr(pk, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pk, "_lib", None)
    with pytest.raises(ImportError):
        pk.lib()


def test_multicast_check_refuses_host_memory():
    # the cluster-multicast tile loads read only this device's memory: host
    # buffers (and, on a machine without a GPU, anything) are refused
    pk = pytest.importorskip("sparse_top_lookup_gb300")
    import ctypes
    import numpy as np
    L = pk.lib()
    a, b = np.zeros(64, np.uint16), np.zeros(64, np.uint16)
    ptrs = (ctypes.c_void_p * 2)(a.ctypes.data, b.ctypes.data)
    assert L.pkm_multicast_ok(ptrs, 2) == 0
    assert L.pkm_multicast_ok(None, 1) == 0
    empty = (ctypes.c_void_p * 1)(None)
    assert L.pkm_multicast_ok(empty, 1) == 0
