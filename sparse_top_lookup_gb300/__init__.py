"""Python binding of the PKM lookup C ABI (include/pkm.h).

Argument marshalling only: every step of the lookup runs in the CUDA kernels
of libpkm.so.  Tensor arguments may be torch tensors (their data_ptr is
passed), numpy arrays (host memory, for pkm_forward_host), raw integer
addresses, or None for optional outputs.  There is no CPU fallback: if
libpkm.so has not been built, importing the library handle raises.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkm.so")
INCLUDE = os.path.join(os.path.dirname(_HERE), "include", "pkm.h")

PKM_F32, PKM_BF16, PKM_FP8_E4M3 = 0, 1, 2
PKM_OK = 0
PKM_ERR_INVALID, PKM_ERR_RANGE, PKM_ERR_UNSUPPORTED, PKM_ERR_ALIGN = -1, -2, -3, -4
PKM_ERR_CUDA, PKM_ERR_NOMEM, PKM_ERR_TIMEOUT, PKM_ERR_BAD_INDEX = -5, -6, -7, -8
PKM_ERR_NO_STAGING, PKM_ERR_OPTION, PKM_ERR_NO_BACKWARD = -9, -10, -11
PKM_OPT_HINT_Z, PKM_OPT_HOST_CHUNKS, PKM_OPT_TEST_STALL = 1, 2, 3
PKM_OPT_READ_SMS = 4
PKM_OPT_SELECT_FORM = 5
PKM_HOST_MAX_CHUNKS = 16

EXPORTED = ["pkm_create", "pkm_destroy", "pkm_forward", "pkm_lookup", "pkm_gather",
            "pkm_forward_host", "pkm_get_status", "pkm_check_args", "pkm_strerror",
            "pkm_abi_version", "pkm_set_option", "pkm_get_fallback_count", "pkm_lookup_static",
            "pkm_quantize_values_fp8", "pkm_bn_fold", "pkm_query_net", "pkm_backward", "pkm_backward_read",
            "pkm_backward_scores", "pkm_forward_host_async", "pkm_backward_sparse",
            "pkm_backward_read_sparse", "pkm_multicast_ok", "pkm_full_keys", "pkm_flat_lookup",
            "pkm_query_net_batch", "pkm_query_net_batch_workspace_bytes"]
PKM_STATIC_MAX_PAIRS = 1 << 16


class pkm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("d_q", "d_v", "max_B", "max_H", "max_n_keys", "max_k", "q_dtype", "key_dtype",
                 "value_dtype", "host_staging", "with_backward")]


class PkmError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, pkm_strerror(code), code))


def build(force=False):
    """Compile libpkm.so for sm_103a (nvcc)."""
    from . import builder as _b
    return _b.build(force=force)


_lib = None


def lib():
    """The loaded libpkm.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libpkm.so is not built (run sparse_top_lookup_gb300.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        cfgp = ctypes.POINTER(pkm_config)
        L.pkm_create.argtypes = [ctypes.POINTER(vp), cfgp]
        L.pkm_destroy.argtypes = [vp]
        L.pkm_destroy.restype = None
        L.pkm_forward.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.pkm_lookup.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.pkm_gather.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.pkm_forward_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.pkm_forward_host_async.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp,
                                             vp]
        L.pkm_get_status.argtypes = [vp, vp]
        L.pkm_check_args.argtypes = [cfgp, i32, i32, i32, i32]
        L.pkm_strerror.argtypes = [i32]
        L.pkm_strerror.restype = ctypes.c_char_p
        L.pkm_abi_version.argtypes = []
        L.pkm_set_option.argtypes = [vp, i32, ctypes.c_double]
        L.pkm_lookup_static.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
        L.pkm_get_fallback_count.argtypes = [vp, vp, ctypes.POINTER(i32)]
        L.pkm_quantize_values_fp8.argtypes = [vp, i32, ctypes.c_int64, i32, vp, vp]
        L.pkm_bn_fold.argtypes = [vp, vp, vp, vp, ctypes.c_float, i32, vp, vp, vp]
        L.pkm_query_net.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.pkm_backward.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.pkm_backward_read.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.pkm_backward_scores.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.pkm_backward_sparse.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp]
        L.pkm_full_keys.argtypes = [vp, vp, i32, i32, vp, vp]
        L.pkm_query_net_batch.argtypes = [vp, vp, i32, i32, i32, vp, vp, ctypes.c_float, vp, vp,
                                          vp, vp, vp, vp]
        L.pkm_query_net_batch_workspace_bytes.argtypes = [i32, i32]
        L.pkm_query_net_batch_workspace_bytes.restype = ctypes.c_size_t
        L.pkm_flat_lookup.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.pkm_backward_read_sparse.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                               vp, vp, vp]
        for f in ("pkm_create", "pkm_forward", "pkm_lookup", "pkm_gather", "pkm_forward_host",
                  "pkm_get_status", "pkm_check_args", "pkm_abi_version", "pkm_set_option",
                  "pkm_get_fallback_count", "pkm_lookup_static", "pkm_quantize_values_fp8",
                  "pkm_bn_fold", "pkm_query_net", "pkm_backward", "pkm_backward_read",
                  "pkm_backward_scores", "pkm_forward_host_async", "pkm_backward_sparse",
                  "pkm_backward_read_sparse", "pkm_full_keys", "pkm_flat_lookup",
                  "pkm_query_net_batch"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _addr(x):
    """Device or host address of a tensor / array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("cannot take the address of %r" % type(x))


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_config(d_q, d_v, max_B, max_H, max_n_keys, max_k, q_dtype=PKM_BF16, key_dtype=None,
                value_dtype=None, host_staging=0, with_backward=0):
    key_dtype = q_dtype if key_dtype is None else key_dtype
    value_dtype = q_dtype if value_dtype is None else value_dtype
    return pkm_config(d_q, d_v, max_B, max_H, max_n_keys, max_k, q_dtype, key_dtype, value_dtype,
                      int(bool(host_staging)), int(bool(with_backward)))


def pkm_strerror(code):
    return lib().pkm_strerror(code).decode()


def pkm_abi_version():
    return lib().pkm_abi_version()


def pkm_check_args(cfg, B, H, n_keys, k):
    return lib().pkm_check_args(ctypes.byref(cfg), B, H, n_keys, k)


def pkm_create(cfg):
    h = ctypes.c_void_p()
    rc = lib().pkm_create(ctypes.byref(h), ctypes.byref(cfg))
    if rc != PKM_OK:
        raise PkmError(rc, "pkm_create")
    return h


def pkm_destroy(h):
    lib().pkm_destroy(h)


def pkm_forward(h, q, subkeys, values, B, H, n_keys, k, out, idx=None, w=None, stream=None):
    return lib().pkm_forward(h, _addr(q), _addr(subkeys), _addr(values), B, H, n_keys, k,
                             _addr(out), _addr(idx), _addr(w), _stream(stream))


def pkm_lookup(h, q, subkeys, B, H, n_keys, k, idx, w, stream=None):
    return lib().pkm_lookup(h, _addr(q), _addr(subkeys), B, H, n_keys, k, _addr(idx), _addr(w),
                            _stream(stream))


def pkm_full_keys(h, subkeys, H, n_keys, keys, stream=None):
    """The full key table [H][n_keys^2][d_q] from the subkeys (see include/pkm.h)."""
    return lib().pkm_full_keys(h, _addr(subkeys), H, n_keys, _addr(keys), _stream(stream))


def pkm_flat_lookup(h, q, keys, B, H, n_keys, k, idx, w, stream=None):
    """Top-k over all n_keys^2 full keys and its softmax (see include/pkm.h)."""
    return lib().pkm_flat_lookup(h, _addr(q), _addr(keys), B, H, n_keys, k, _addr(idx), _addr(w),
                                 _stream(stream))


def pkm_gather(h, values, B, H, n_keys, k, idx, w, out, stream=None):
    return lib().pkm_gather(h, _addr(values), B, H, n_keys, k, _addr(idx), _addr(w), _addr(out),
                            _stream(stream))


def pkm_backward(h, q, subkeys, values, B, H, n_keys, k, idx, w, dout, dq, dsubkeys, dvalues,
                 stream=None):
    """Gradients of pkm_forward for its selection: dq overwritten, dsubkeys and dvalues added to."""
    return lib().pkm_backward(h, _addr(q), _addr(subkeys), _addr(values), B, H, n_keys, k,
                              _addr(idx), _addr(w), _addr(dout), _addr(dq), _addr(dsubkeys),
                              _addr(dvalues), _stream(stream))


def pkm_backward_sparse(h, q, subkeys, values, B, H, n_keys, k, idx, w, dout, dq, dsubkeys, rows,
                        grad_rows, n_rows, stream=None):
    """Gradients with the value-table part sparse: rows[:n_rows] (distinct, ascending) and
    grad_rows[:n_rows]; n_rows is a device int32."""
    return lib().pkm_backward_sparse(h, _addr(q), _addr(subkeys), _addr(values), B, H, n_keys, k,
                                     _addr(idx), _addr(w), _addr(dout), _addr(dq),
                                     _addr(dsubkeys), _addr(rows), _addr(grad_rows),
                                     _addr(n_rows), _stream(stream))


def pkm_backward_read_sparse(h, values, B, H, n_keys, k, idx, w, dout, dw, rows, grad_rows, n_rows,
                             stream=None):
    """dw and the sparse value-table gradient (see pkm_backward_sparse)."""
    return lib().pkm_backward_read_sparse(h, _addr(values), B, H, n_keys, k, _addr(idx), _addr(w),
                                          _addr(dout), _addr(dw), _addr(rows), _addr(grad_rows),
                                          _addr(n_rows), _stream(stream))


def pkm_backward_read(h, values, B, H, n_keys, k, idx, w, dout, dw, dvalues, stream=None):
    """dw = dout . V[idx] (overwritten) and dvalues[idx] += w * dout."""
    return lib().pkm_backward_read(h, _addr(values), B, H, n_keys, k, _addr(idx), _addr(w),
                                   _addr(dout), _addr(dw), _addr(dvalues), _stream(stream))


def pkm_backward_scores(h, q, subkeys, B, H, n_keys, k, idx, w, dw, dq, dsubkeys, stream=None):
    """dq (overwritten) and dsubkeys (added to) from the weights and their gradient dw."""
    return lib().pkm_backward_scores(h, _addr(q), _addr(subkeys), B, H, n_keys, k, _addr(idx),
                                     _addr(w), _addr(dw), _addr(dq), _addr(dsubkeys),
                                     _stream(stream))


def pkm_forward_host(h, q_host, subkeys, values, B, H, n_keys, k, out_host, idx_host=None,
                     w_host=None, stream=None):
    return lib().pkm_forward_host(h, _addr(q_host), _addr(subkeys), _addr(values), B, H, n_keys, k,
                                  _addr(out_host), _addr(idx_host), _addr(w_host),
                                  _stream(stream))


def pkm_forward_host_async(h, q_host, subkeys, values, B, H, n_keys, k, out_host, done_event,
                           idx_host=None, w_host=None, stream=None):
    """pkm_forward_host without the final synchronisation; done_event (a
    torch.cuda.Event or a raw cudaEvent_t) completes when the results are
    back in the host buffers."""
    if hasattr(done_event, "cuda_event"):
        if not done_event.cuda_event:  # torch creates its events when first recorded
            done_event.record()
        ev = done_event.cuda_event
    else:
        ev = done_event
    return lib().pkm_forward_host_async(h, _addr(q_host), _addr(subkeys), _addr(values), B, H,
                                        n_keys, k, _addr(out_host), _addr(idx_host),
                                        _addr(w_host), _stream(stream), ev)


def pkm_set_option(h, option, value):
    return lib().pkm_set_option(h, option, float(value))


def pkm_get_fallback_count(h, stream=None):
    """Pairs of the last bf16 lookup whose threshold hint missed (re-selected; synchronises)."""
    c = ctypes.c_int()
    check(lib().pkm_get_fallback_count(h, _stream(stream), ctypes.byref(c)),
          "pkm_get_fallback_count")
    return c.value


def pkm_lookup_static(q, subkeys, B, H, d_q, n_keys, k, idx, w, status=None, stream=None):
    """The bf16 lookup without a handle or any device allocation (see include/pkm.h)."""
    return lib().pkm_lookup_static(_addr(q), _addr(subkeys), B, H, d_q, n_keys, k, _addr(idx),
                                   _addr(w), _addr(status), _stream(stream))


def pkm_query_net_batch_workspace_bytes(B, F):
    return int(lib().pkm_query_net_batch_workspace_bytes(B, F))


def pkm_query_net_batch(x, weight, B, dim, F, gamma, beta, eps, workspace, q, batch_mean=None,
                        batch_var=None, status=None, stream=None):
    """The query network with the batch's own BatchNorm statistics (see include/pkm.h)."""
    return lib().pkm_query_net_batch(_addr(x), _addr(weight), B, dim, F, _addr(gamma),
                                     _addr(beta), float(eps), _addr(workspace), _addr(q),
                                     _addr(batch_mean), _addr(batch_var), _addr(status),
                                     _stream(stream))


def pkm_quantize_values_fp8(values, value_dtype, N, d_v, out, stream=None):
    """Write the fp8 e4m3 table (N*d_v codes, then N fp32 scales) of an fp32/bf16 table."""
    return lib().pkm_quantize_values_fp8(_addr(values), value_dtype, N, d_v, _addr(out),
                                         _stream(stream))


def pkm_bn_fold(gamma, beta, running_mean, running_var, eps, F, scale, shift, stream=None):
    """Per-feature scale / shift of an eval-mode BatchNorm1d (device arrays)."""
    return lib().pkm_bn_fold(_addr(gamma), _addr(beta), _addr(running_mean), _addr(running_var),
                             float(eps), F, _addr(scale), _addr(shift), _stream(stream))


def pkm_query_net(x, weight, B, dim, F, scale, shift, q, status=None, stream=None):
    """q = (x W^T) * scale + shift in bf16: the query network ahead of the lookup."""
    return lib().pkm_query_net(_addr(x), _addr(weight), B, dim, F, _addr(scale), _addr(shift),
                               _addr(q), _addr(status), _stream(stream))


def fp8_table_bytes(N, d_v):
    """Size of the PKM_FP8_E4M3 value buffer: codes then row scales."""
    return N * d_v + 4 * N


def pkm_get_status(h, stream=None):
    return lib().pkm_get_status(h, _stream(stream))


def check(rc, where):
    """Raise PkmError unless rc is PKM_OK."""
    if rc != PKM_OK:
        raise PkmError(rc, where)
