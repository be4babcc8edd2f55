"""The fp8 e4m3 value table on the GPU, against the fp64 oracle.

Product-Key Memory, note after the code listing: the value table is "a good
candidate for keeping in a lower precision".  Layout: N rows of e4m3 codes
then N fp32 row scales.  The quantiser is compared bit for bit with the
oracle's (the same fp32 division and nearest-even rounding decide every
code); the fp8 read and the whole forward pass are compared with the
oracle's exact fp64 read of the oracle-quantised table.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, compare_lookup, compare_out

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")


def dev_bits(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def to_bf16(x):
    """float32 -> bf16 bits, round to nearest even (torch's conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def packed_table(codes, scales):
    """The PKM_FP8_E4M3 buffer (codes, then scales) on the device."""
    buf = np.concatenate([codes.reshape(-1), scales.view(np.uint8)])
    return torch.from_numpy(buf).cuda()


def gpu_quantize(V, N, d_v, dtype):
    out = torch.empty(pk.fp8_table_bytes(N, d_v), dtype=torch.uint8, device="cuda")
    pk.check(pk.pkm_quantize_values_fp8(dev_bits(V), dtype, N, d_v, out), "quantize")
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    return o[: N * d_v].reshape(N, d_v), o[N * d_v:].view(np.float32)


def test_quantiser_matches_oracle_bit_for_bit():
    rng = np.random.default_rng(21)
    for N, d_v, dtype in ((257, 64, pk.PKM_BF16), (100, 1024, pk.PKM_BF16),
                          (64, 48, pk.PKM_F32)):
        V = rng.standard_normal((N, d_v)) * rng.choice([1e-38, 1e-20, 1e-3, 1.0, 3e4], (N, 1))
        V[3] = 0.0
        V[4] = 0.0
        V[4, d_v - 1] = -7.0
        V[5, ::7] = 448.0 * 3                   # many elements tied at amax
        if dtype == pk.PKM_BF16:
            Vb = to_bf16(V)
        else:
            Vb = V.astype(np.float32)
        codes, scales = gpu_quantize(Vb, N, d_v, dtype)
        rc, rs = oracle.quantize_fp8(Vb, N, d_v)
        assert (scales.view(np.uint32) == rs.view(np.uint32)).all(), (N, d_v)
        assert (codes == rc).all(), (N, d_v, np.argwhere(codes != rc)[:5])


def test_fp8_gather_matches_oracle():
    rng = np.random.default_rng(22)
    N, d_v, B, H, k = 4096, 256, 300, 3, 16
    V = synth.normal(22, 3, N * d_v, 1.0 / d_v, dtype="bf16").reshape(N, d_v)
    codes, scales = oracle.quantize_fp8(V, N, d_v)
    table = packed_table(codes, scales)
    idx = rng.integers(0, N, (B, H, k)).astype(np.int64)
    w = rng.random((B, H, k)).astype(np.float32)
    w /= w.sum(-1, keepdims=True)
    n = 64  # N = n_keys^2
    cfg = pk.make_config(128, d_v, B, H, n, k, q_dtype=pk.PKM_BF16, value_dtype=pk.PKM_FP8_E4M3)
    h = pk.pkm_create(cfg)
    try:
        out = torch.empty(B, d_v, device="cuda")
        pk.check(pk.pkm_gather(h, table, B, H, n, k, torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w).cuda(), out), "gather")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        got = out.cpu().numpy().astype(np.float64)
        # a planted out-of-range index is skipped and reported
        bad = idx.copy()
        bad[0, 0, 0] = N
        out2 = torch.empty(B, d_v, device="cuda")
        pk.check(pk.pkm_gather(h, table, B, H, n, k, torch.from_numpy(bad).cuda(),
                               torch.from_numpy(w).cuda(), out2), "gather")
        assert pk.pkm_get_status(h) == pk.PKM_ERR_BAD_INDEX
    finally:
        pk.pkm_destroy(h)
    ref = oracle.gather_fp8(codes, scales, N, d_v, idx, w.astype(np.float64))
    err = np.abs(got - ref) / (1 + np.abs(ref))
    assert err.max() <= TOL, err.max()


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, d_v, k
    (300, 2, 128, 256, 128, 16),
    (129, 2, 1024, 1024, 1024, 32),  # page-width rows, small batch
])
def test_forward_with_fp8_table_matches_oracle(shape):
    B, H, d_q, n, d_v, k = shape
    seed = sum(shape)
    q = synth.normal(seed, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(seed, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    N = n * n
    V = synth.normal(seed, 3, N * d_v, 1.0 / d_v, dtype="bf16").reshape(N, d_v)
    codes, scales = oracle.quantize_fp8(V, N, d_v)
    table = packed_table(codes, scales)
    cfg = pk.make_config(d_q, d_v, B, H, n, k, q_dtype=pk.PKM_BF16, value_dtype=pk.PKM_FP8_E4M3)
    h = pk.pkm_create(cfg)
    try:
        out = torch.empty(B, d_v, device="cuda")
        idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w = torch.empty(B, H, k, device="cuda")
        pk.check(pk.pkm_forward(h, dev_bits(q), dev_bits(C), table, B, H, n, k, out, idx, w),
                 "forward")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        gout, gidx, gw = out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    finally:
        pk.pkm_destroy(h)
    ref = oracle.lookup(q, C, B, H, d_q, n, k)
    rep = compare_lookup(gidx, gw, ref, q, C, "bf16", H, d_q, n)
    assert rep["failures"] == 0, rep
    ref_out = oracle.gather_fp8(codes, scales, N, d_v, ref["idx"], ref["w"])
    err = compare_out(gout, None, N, d_v, gidx, ref["idx"], ref["w"], ref_out,
                      regather=lambda i, ww: oracle.gather_fp8(codes, scales, N, d_v, i, ww))
    assert err <= TOL, err
