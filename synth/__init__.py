"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

Only random-number generation lives here (see gen.c for the exact
definition of every stream); none of the lookup arithmetic does.  Arrays are
returned as numpy: fp32 as float32, bf16 as raw uint16 bit patterns.
"""
import ctypes
import math
import os
import subprocess

import numpy as np

from .configs import (CONFIGS, TID_BN, TID_KEYS, TID_MIX_MEAN, TID_MIX_PICK, TID_Q, TID_QW,
                      TID_SEL, TID_VALUES, TID_X, n_rows, seed_of)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    """Compile gen.c into libsynth.so (plain C, host only)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm", "-lpthread"])
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, f64, i32, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                  ctypes.c_int, ctypes.c_void_p)
        L.synth_normal_f32.argtypes = [u64, u64, i64, i64, f64, f64, vp, i32]
        L.synth_normal_bf16.argtypes = [u64, u64, i64, i64, f64, f64, vp, i32]
        L.synth_uniform_f64.argtypes = [u64, u64, i64, i64, vp, i32]
        L.synth_mixture_bf16.argtypes = [u64, u64, u64, u64, i64, i64, i64, i32, f64, f64, vp,
                                         vp, i32]
        L.synth_mixture_bf16.restype = i32
        L.synth_f32_to_bf16.argtypes = [vp, vp, i64]
        L.synth_draw_u64.argtypes = [u64, u64, u64]
        L.synth_draw_u64.restype = u64
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def normal(seed, tensor_id, n, var=1.0, mean=0.0, dtype="f32", offset=0, nthreads=0):
    """Elements [offset, offset+n) of stream (seed, tensor_id) drawn N(mean, var)."""
    sd = math.sqrt(var)
    if dtype == "f32":
        out = np.empty(n, np.float32)
        lib().synth_normal_f32(seed, tensor_id, offset, n, mean, sd, _ptr(out), nthreads)
    elif dtype == "bf16":
        out = np.empty(n, np.uint16)
        lib().synth_normal_bf16(seed, tensor_id, offset, n, mean, sd, _ptr(out), nthreads)
    else:
        raise ValueError(dtype)
    return out


def uniform(seed, tensor_id, n, offset=0, nthreads=0):
    out = np.empty(n, np.float64)
    lib().synth_uniform_f64(seed, tensor_id, offset, n, _ptr(out), nthreads)
    return out


def mixture_bf16(seed, row_len, rows, n_comp, zipf_s, comp_sd, row_offset=0, nthreads=0,
                 with_components=False):
    out = np.empty(rows * row_len, np.uint16)
    comp = np.empty(rows, np.int32) if with_components else None
    rc = lib().synth_mixture_bf16(seed, TID_Q, TID_MIX_MEAN, TID_MIX_PICK, row_len,
                                  row_offset * row_len, rows * row_len, n_comp, zipf_s, comp_sd,
                                  _ptr(out), _ptr(comp) if comp is not None else None, nthreads)
    if rc != 0:
        raise ValueError("mixture arguments rejected (%d)" % rc)
    return (out, comp) if with_components else out


def f32_to_bf16(x):
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().synth_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(u):
    """Exact widening of raw bf16 bits to float32."""
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ workloads

def queries(cfg, rows=None, row_offset=0):
    """q [rows, H, d_q] (flattened) for queries row_offset .. row_offset+rows."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rows = cfg["B"] if rows is None else rows
    row_len = cfg["H"] * cfg["d_q"]
    if cfg["q_kind"] == "mixture":
        return mixture_bf16(seed_of(cfg), row_len, rows, cfg["mix_components"],
                            cfg["mix_zipf_s"], cfg["mix_sd"], row_offset=row_offset)
    return normal(seed_of(cfg), TID_Q, rows * row_len, cfg["q_var"], dtype=cfg["dtype"],
                  offset=row_offset * row_len)


def subkeys(cfg):
    """subkeys [H, 2, n_keys, d_q/2] (flattened)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    n = cfg["H"] * 2 * cfg["n_keys"] * (cfg["d_q"] // 2)
    return normal(seed_of(cfg), TID_KEYS, n, cfg["key_var"], dtype=cfg["dtype"])


def values(cfg, nthreads=0):
    """value table [n_keys**2, d_v] (flattened)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    n = n_rows(cfg) * cfg["d_v"]
    return normal(seed_of(cfg), TID_VALUES, n, cfg["value_var"], dtype=cfg["dtype"],
                  nthreads=nthreads)


def value_rows(cfg, rows):
    """Selected rows of the value table, [len(rows), d_v], without building it all."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    d = cfg["d_v"]
    out = np.empty((len(rows), d), np.float32 if cfg["dtype"] == "f32" else np.uint16)
    for i, r in enumerate(rows):
        out[i] = normal(seed_of(cfg), TID_VALUES, d, cfg["value_var"], dtype=cfg["dtype"],
                        offset=int(r) * d, nthreads=1)
    return out


def query_net_inputs(cfg, rows=None, row_offset=0):
    """Query-network inputs of a layer workload: x [rows, dim] bf16 bits,
    W [H*d_q, dim] bf16 bits, and the BatchNorm's gamma ~ 1 + N(0, 0.01),
    beta ~ N(0, 0.01), running mean ~ N(0, 0.0025), running var ~ 1 + |N(0, 0.01)|
    (fp32, one per feature)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rows = cfg["B"] if rows is None else rows
    dim, F, s = cfg["qnet_dim"], cfg["H"] * cfg["d_q"], seed_of(cfg)
    x = normal(s, TID_X, rows * dim, 1.0, dtype="bf16", offset=row_offset * dim)
    W = normal(s, TID_QW, F * dim, 1.0 / dim, dtype="bf16")
    gamma = normal(s, TID_BN, F, 0.01, mean=1.0)
    beta = normal(s, TID_BN + 1, F, 0.01)
    mean = normal(s, TID_BN + 2, F, 0.0025)
    var = (1.0 + np.abs(normal(s, TID_BN + 3, F, 0.01))).astype(np.float32)
    return x, W, gamma, beta, mean, var


def selections(cfg, rows=None, row_offset=0):
    """A stand-in selection for backward-pass inputs, shaped like a lookup's:
    per (query, head), S = ceil(sqrt(2k)) subkeys drawn uniformly for each
    half, then k winners, each a uniform pick of one subkey from each half's
    list (so winners share subkeys, as selected keys do; a winner may repeat,
    which a lookup never gives but the gradient sums alike), and positive weights
    summing to 1 (exponential draws, normalised; flat Dirichlet).  Returns
    (a1, a2, w): [rows, H, k] int64 subkey numbers and float32 weights."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rows = cfg["B"] if rows is None else rows
    H, n, k, s = cfg["H"], cfg["n_keys"], cfg["k"], seed_of(cfg)
    S = min(n, int(math.ceil(math.sqrt(2 * k))))
    P = rows * H
    lists = uniform(s, TID_SEL, P * 2 * S, offset=row_offset * H * 2 * S).reshape(P, 2, S)
    lists = np.minimum((lists * n).astype(np.int64), n - 1)
    pick = uniform(s, TID_SEL + 1, P * 2 * k, offset=row_offset * H * 2 * k).reshape(P, 2, k)
    pick = np.minimum((pick * S).astype(np.int64), S - 1)
    a1 = np.take_along_axis(lists[:, 0], pick[:, 0], axis=1)
    a2 = np.take_along_axis(lists[:, 1], pick[:, 1], axis=1)
    e = -np.log1p(-uniform(s, TID_SEL + 2, P * k, offset=row_offset * H * k)).reshape(P, k)
    w = (e / e.sum(1, keepdims=True)).astype(np.float32)
    return a1.reshape(rows, H, k), a2.reshape(rows, H, k), w.reshape(rows, H, k)


def output_grads(cfg, rows=None, row_offset=0):
    """dout [rows, d_v] float32 ~ N(0, 1): the gradient arriving at the read's output."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rows = cfg["B"] if rows is None else rows
    d = cfg["d_v"]
    return normal(seed_of(cfg), TID_SEL + 3, rows * d, 1.0, offset=row_offset * d).reshape(rows, d)


__all__ = ["CONFIGS", "build", "normal", "uniform", "mixture_bf16", "f32_to_bf16",
           "bf16_to_f32", "queries", "subkeys", "values", "value_rows", "seed_of", "n_rows",
           "query_net_inputs", "selections", "output_grads"]
