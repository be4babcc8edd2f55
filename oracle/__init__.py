"""Python handle on the fp64 CPU oracle (pkm_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests, by the package smoke check and
by the benchmark's CPU-baseline leg, never by the product path.  Inputs are
numpy arrays: float32, or uint16 holding raw bf16 bits.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkm_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, BF16 = 0, 1


def build(force=False):
    """Compile the oracle with g++ (OpenMP over independent queries if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp, _SRC]
    try:
        subprocess.check_call(base + ["-fopenmp"], stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.check_call(base)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.oracle_lookup.argtypes = [vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                    vp, i32]
        L.oracle_gather.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, i32]
        L.oracle_forward.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, vp,
                                     vp, vp, i32]
        L.oracle_brute_topk.argtypes = [vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, i32]
        L.oracle_quantize_fp8.argtypes = [vp, i32, i64, i32, vp, vp, i32]
        L.oracle_backward.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                      vp, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_query_net.argtypes = [vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp,
                                       ctypes.c_double, vp, i32]
        L.oracle_query_net_batch.argtypes = [vp, i32, vp, i32, i32, i32, i32, vp, vp,
                                             ctypes.c_double, vp, vp, vp, i32]
        L.oracle_gather_fp8.argtypes = [vp, vp, i64, i32, i32, i32, i32, vp, vp, vp, i32]
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        for f in (L.oracle_lookup, L.oracle_gather, L.oracle_forward, L.oracle_brute_topk,
                  L.oracle_num_threads, L.oracle_quantize_fp8, L.oracle_gather_fp8,
                  L.oracle_query_net, L.oracle_query_net_batch, L.oracle_backward):
            f.restype = i32
        _lib = L
    return _lib


def _dt(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("oracle inputs are float32 or uint16 (bf16 bits), got %s" % a.dtype)


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a):
    return np.ascontiguousarray(a)


def num_threads():
    return lib().oracle_num_threads()


def lookup(q, subkeys, B, H, d_q, n_keys, k, want_gaps=False, nthreads=0):
    """Steps up to the softmax.  Returns dict(idx, score, w[, gap_k, gap_in, counters])."""
    q, subkeys = _c(q), _c(subkeys)
    idx = np.empty((B, H, k), np.int64)
    score = np.empty((B, H, k), np.float64)
    w = np.empty((B, H, k), np.float64)
    gap_k = np.empty((B, H), np.float64) if want_gaps else None
    gap_in = np.empty((B, H), np.float64) if want_gaps else None
    counters = np.zeros(2, np.int64)
    rc = lib().oracle_lookup(_p(q), _dt(q), _p(subkeys), _dt(subkeys), B, H, d_q, n_keys, k,
                             _p(idx), _p(score), _p(w), _p(gap_k), _p(gap_in), _p(counters),
                             nthreads)
    if rc != 0:
        raise ValueError("oracle_lookup rejected the shape (B=%d H=%d d_q=%d n=%d k=%d)"
                         % (B, H, d_q, n_keys, k))
    out = dict(idx=idx, score=score, w=w, counters=counters)
    if want_gaps:
        out.update(gap_k=gap_k, gap_in=gap_in)
    return out


def gather(values, N, d_v, idx, w, nthreads=0):
    """out[b] = sum_{h,j} w[b,h,j] * V[idx[b,h,j]] in double."""
    values = _c(values)
    idx = np.ascontiguousarray(idx, np.int64)
    w = np.ascontiguousarray(w, np.float64)
    B, H, k = idx.shape
    out = np.empty((B, d_v), np.float64)
    rc = lib().oracle_gather(_p(values), _dt(values), N, d_v, B, H, k, _p(idx), _p(w), _p(out),
                             nthreads)
    if rc != 0:
        raise ValueError("oracle_gather: bad shape or index out of range")
    return out


def forward(q, subkeys, values, B, H, d_q, n_keys, d_v, k, nthreads=0):
    """Whole forward pass.  Returns (idx, w, out)."""
    q, subkeys, values = _c(q), _c(subkeys), _c(values)
    idx = np.empty((B, H, k), np.int64)
    w = np.empty((B, H, k), np.float64)
    out = np.empty((B, d_v), np.float64)
    rc = lib().oracle_forward(_p(q), _dt(q), _p(subkeys), _dt(subkeys), _p(values), _dt(values),
                              B, H, d_q, n_keys, d_v, k, _p(idx), _p(w), _p(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return idx, w, out


def brute_topk(q, subkeys, B, H, d_q, n_keys, k, nthreads=0):
    """Top-k over all n_keys**2 full keys, each scored as one d_q-long dot product."""
    q, subkeys = _c(q), _c(subkeys)
    idx = np.empty((B, H, k), np.int64)
    score = np.empty((B, H, k), np.float64)
    rc = lib().oracle_brute_topk(_p(q), _dt(q), _p(subkeys), _dt(subkeys), B, H, d_q, n_keys, k,
                                 _p(idx), _p(score), nthreads)
    if rc != 0:
        raise ValueError("oracle_brute_topk rejected the shape")
    return idx, score


def e4m3_value(code):
    """The value of one fp8 e4m3 code (format definition)."""
    return lib().oracle_e4m3_value(int(code))


def e4m3_encode(x):
    """The e4m3 code nearest to the float32 x (ties to even, saturated)."""
    return int(lib().oracle_e4m3_encode(float(np.float32(x))))


def quantize_fp8(values, N, d_v, nthreads=0):
    """Per-row fp8 e4m3 quantisation.  Returns (codes uint8 [N, d_v], scales float32 [N])."""
    values = _c(values)
    codes = np.empty((N, d_v), np.uint8)
    scales = np.empty(N, np.float32)
    rc = lib().oracle_quantize_fp8(_p(values), _dt(values), N, d_v, _p(codes), _p(scales),
                                   nthreads)
    if rc != 0:
        raise ValueError("oracle_quantize_fp8: bad shape")
    return codes, scales


def gather_fp8(codes, scales, N, d_v, idx, w, nthreads=0):
    """out[b] = sum_{h,j} w[b,h,j] * scale[r] * value(codes[r]) in double, r = idx[b,h,j]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    idx = np.ascontiguousarray(idx, np.int64)
    w = np.ascontiguousarray(w, np.float64)
    B, H, k = idx.shape
    out = np.empty((B, d_v), np.float64)
    rc = lib().oracle_gather_fp8(_p(codes), _p(scales), N, d_v, B, H, k, _p(idx), _p(w), _p(out),
                                 nthreads)
    if rc != 0:
        raise ValueError("oracle_gather_fp8: bad shape or index out of range")
    return out


def query_net(x, weight, B, dim, F, gamma, beta, mean, var, eps, nthreads=0):
    """q = BatchNorm1d(x W^T) with running statistics, in double.  Returns [B, F]."""
    x, weight = _c(x), _c(weight)
    params = [np.ascontiguousarray(a, np.float32) for a in (gamma, beta, mean, var)]
    q = np.empty((B, F), np.float64)
    rc = lib().oracle_query_net(_p(x), _dt(x), _p(weight), _dt(weight), B, dim, F,
                                *[_p(a) for a in params], float(eps), _p(q), nthreads)
    if rc != 0:
        raise ValueError("oracle_query_net: bad shape")
    return q


def query_net_batch(x, weight, B, dim, F, gamma, beta, eps, nthreads=0):
    """q = BatchNorm1d(x W^T) normalised by the batch's own statistics (training
    mode), in double.  Returns (q [B, F], batch mean [F], biased batch variance [F])."""
    x, weight = _c(x), _c(weight)
    g, bt = (np.ascontiguousarray(a, np.float32) for a in (gamma, beta))
    q = np.empty((B, F), np.float64)
    mean = np.empty(F, np.float64)
    var = np.empty(F, np.float64)
    rc = lib().oracle_query_net_batch(_p(x), _dt(x), _p(weight), _dt(weight), B, dim, F, _p(g),
                                      _p(bt), float(eps), _p(q), _p(mean), _p(var), nthreads)
    if rc != 0:
        raise ValueError("oracle_query_net_batch: bad shape")
    return q, mean, var


def backward(q, subkeys, values, B, H, d_q, n_keys, d_v, k, idx, w, dout, dvalue_rows=None):
    """Gradients for a fixed selection.  Returns dict(dw, dq, dsubkeys, dvalues):
    dvalues dense [n_keys**2, d_v] (small problems only), or, with
    dvalue_rows (a list of distinct table rows), [len(dvalue_rows), d_v]
    holding those rows' sums."""
    q, subkeys, values = _c(q), _c(subkeys), _c(values)
    idx = np.ascontiguousarray(idx, np.int64)
    w = np.ascontiguousarray(w, np.float64)
    dout = np.ascontiguousarray(dout, np.float64)
    dw = np.empty((B, H, k), np.float64)
    dq = np.empty((B, H, d_q), np.float64)
    dC = np.zeros((H, 2, n_keys, d_q // 2), np.float64)
    slot = None
    if dvalue_rows is None:
        dV = np.zeros((n_keys * n_keys, d_v), np.float64)
    else:
        rows = np.asarray(dvalue_rows, np.int64)
        slot = np.full(n_keys * n_keys, -1, np.int64)
        slot[rows] = np.arange(len(rows))
        dV = np.zeros((len(rows), d_v), np.float64)
    rc = lib().oracle_backward(_p(q), _dt(q), _p(subkeys), _dt(subkeys), _p(values), _dt(values),
                               B, H, d_q, n_keys, d_v, k, _p(idx), _p(w), _p(dout), _p(dw),
                               _p(dq), _p(dC), _p(dV), None if slot is None else _p(slot))
    if rc != 0:
        raise ValueError("oracle_backward: bad shape or index")
    return dict(dw=dw, dq=dq, dsubkeys=dC, dvalues=dV)
