"""pkm_lookup_static: the bf16 lookup that allocates no device memory.

It serves callers that cannot allocate when they run a lookup (a process
whose GPU memory is budgeted up front, a host framework that owns every
allocation, a hot loop where cudaMalloc / cudaFree would synchronise the
device).  Its scratch is one fixed array in the library; every call reuses
it.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import synth


def test_static_lookup_rejects_too_many_pairs_on_the_host():
    pk = pytest.importorskip("sparse_top_lookup_gb300")
    pk.build()
    L = pk.lib()
    too_many = pk.PKM_STATIC_MAX_PAIRS + 1
    # rejected before any CUDA call: B * H over the fixed scratch size
    assert L.pkm_lookup_static(16, 16, too_many, 1, 64, 64, 4, 16, 16, None, None) \
        == pk.PKM_ERR_RANGE
    assert L.pkm_lookup_static(16, 16, 1, 1, 64, 8, 9, 16, 16, None, None) == pk.PKM_ERR_RANGE
    assert L.pkm_lookup_static(16, 16, 1, 1, 63, 8, 4, 16, 16, None, None) == pk.PKM_ERR_INVALID
    assert L.pkm_lookup_static(16, 16, 1, 1, 72, 8, 4, 16, 16, None, None) \
        == pk.PKM_ERR_UNSUPPORTED


def _static_call(pk, L, q, C, B, H, d_q, n, k):
    """One pkm_lookup_static call through the C ABI; returns idx, w, status."""
    import torch
    idx = torch.full((B, H, k), -7, dtype=torch.int64, device="cuda")
    w = torch.full((B, H, k), -7.0, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.pkm_lookup_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(C.data_ptr()),
                             B, H, d_q, n, k, ctypes.c_void_p(idx.data_ptr()),
                             ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(status.data_ptr()),
                             ctypes.c_void_p(stream))
    assert rc == pk.PKM_OK, pk.pkm_strerror(rc)
    torch.cuda.synchronize()
    return idx, w, status.item()


@pytest.mark.gpu
def test_static_lookup_matches_oracle_and_handle_lookup_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    pk = pytest.importorskip("sparse_top_lookup_gb300")
    import oracle
    from helpers import compare_lookup
    L = pk.lib()

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)

    cases = [  # B, H, d_q, n_keys, k: two calls in a row with different shapes
        (300, 2, 256, 512, 32),
        (130, 3, 128, 256, 16),
    ]
    for seed, (B, H, d_q, n, k) in enumerate(cases, start=41):
        q_np = synth.normal(seed, 1, B * H * d_q, 1.0, dtype="bf16")
        C_np = synth.normal(seed, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
        q, C = dev(q_np), dev(C_np)

        # the existing entry point, through a handle
        h = pk.pkm_create(pk.make_config(d_q, 64, B, H, n, k, q_dtype=pk.PKM_BF16))
        try:
            idx_ref = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
            w_ref = torch.empty(B, H, k, device="cuda")
            pk.check(pk.pkm_lookup(h, q, C, B, H, n, k, idx_ref, w_ref), "pkm_lookup")
            assert pk.pkm_get_status(h) == pk.PKM_OK
        finally:
            pk.pkm_destroy(h)

        # the allocation-free entry point, called through the C ABI directly
        idx, w, st = _static_call(pk, L, q, C, B, H, d_q, n, k)
        assert st == pk.PKM_OK
        assert torch.equal(idx, idx_ref)
        ref = w_ref.double()
        assert ((w.double() - ref).abs() <= 2e-3 * (1 + ref.abs())).all()
        # and against the fp64 oracle, as every other parity test
        want = oracle.lookup(q_np, C_np, B, H, d_q, n, k)
        rep = compare_lookup(idx.cpu().numpy(), w.cpu().numpy(), want, q_np, C_np, "bf16", H,
                             d_q, n)
        assert rep["failures"] == 0 and rep["w_ok"], rep


@pytest.mark.gpu
def test_static_lookup_retry_pass_and_no_allocation():
    # Subkeys that are all equal but for a few make every row's scores a few
    # distinct values above one value shared by all the others: the
    # threshold hint (mean + z * spread) lands above the shared value, every
    # list comes out short, and the retry pass (its counts, unit flags and
    # unit list live in the static array) selects the rows again without the
    # hint, breaking the exact ties by flat index.  Repeated calls leave the
    # device's free memory unchanged.
    torch = pytest.importorskip("torch")
    pk = pytest.importorskip("sparse_top_lookup_gb300")
    import oracle
    L = pk.lib()
    B, H, d_q, n, k = 260, 2, 64, 256, 32
    rng = np.random.default_rng(5)
    qf = rng.integers(-2, 3, (B, H, d_q)).astype(np.float32)
    Cf = np.ones((H, 2, n, d_q // 2), np.float32)
    Cf[:, :, :6] = rng.integers(-2, 3, (H, 2, 6, d_q // 2))
    q_np, C_np = synth.f32_to_bf16(qf).ravel(), synth.f32_to_bf16(Cf).ravel()
    q = torch.from_numpy(q_np.view(np.int16)).cuda().view(torch.bfloat16)
    C = torch.from_numpy(C_np.view(np.int16)).cuda().view(torch.bfloat16)
    want = oracle.lookup(q_np, C_np, B, H, d_q, n, k)
    idx, w, st = _static_call(pk, L, q, C, B, H, d_q, n, k)  # warm-up (and first check)
    assert st == pk.PKM_OK
    assert np.array_equal(idx.cpu().numpy(), want["idx"])
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        idx, w, st = _static_call(pk, L, q, C, B, H, d_q, n, k)
        assert st == pk.PKM_OK
        assert np.array_equal(idx.cpu().numpy(), want["idx"])
        assert (np.abs(w.cpu().numpy() - want["w"]) <= 1e-6 * (1 + want["w"])).all()
    assert torch.cuda.mem_get_info()[0] == free0
    # the same input through a handle shows that the lists did go through
    # the retry pass
    h = pk.pkm_create(pk.make_config(d_q, 64, B, H, n, k, q_dtype=pk.PKM_BF16))
    try:
        i2 = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w2 = torch.empty(B, H, k, device="cuda")
        pk.check(pk.pkm_lookup(h, q, C, B, H, n, k, i2, w2), "pkm_lookup")
        assert pk.pkm_get_fallback_count(h) > 0
        assert torch.equal(i2, idx)
    finally:
        pk.pkm_destroy(h)


@pytest.mark.gpu
def test_handle_calls_do_not_allocate_after_warm_up():
    # pkm_create is the only call that allocates: after one warm-up call of
    # each entry point (which may load kernels), repeated calls leave the
    # device's free memory unchanged
    torch = pytest.importorskip("torch")
    pk = pytest.importorskip("sparse_top_lookup_gb300")
    B, H, d_q, n, d_v, k = 256, 2, 128, 128, 128, 16
    s = 55

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)

    q_np = synth.normal(s, 1, B * H * d_q, 1.0, dtype="bf16")
    q, C = dev(q_np), dev(synth.normal(s, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16"))
    V = dev(synth.normal(s, 3, n * n * d_v, 1.0 / d_v, dtype="bf16"))
    cfg = pk.make_config(d_q, d_v, B, H, n, k, q_dtype=pk.PKM_BF16, host_staging=1,
                         with_backward=1)
    h = pk.pkm_create(cfg)
    try:
        out = torch.empty(B, d_v, device="cuda")
        idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w = torch.empty(B, H, k, device="cuda")
        dout = torch.randn(B, d_v, device="cuda", generator=torch.Generator("cuda").manual_seed(1))
        dq = torch.empty(B, H, d_q, device="cuda")
        dC = torch.zeros(H, 2, n, d_q // 2, device="cuda")
        dVt = torch.zeros(n * n, d_v, device="cuda")
        rows = torch.empty(B * H * k, dtype=torch.int64, device="cuda")
        grad = torch.empty(B * H * k, d_v, device="cuda")
        nr = torch.zeros(1, dtype=torch.int32, device="cuda")
        qh = torch.from_numpy(q_np.view(np.int16)).pin_memory()
        oh = torch.empty(B, d_v).pin_memory()
        ev = torch.cuda.Event()

        def round_of_calls():
            pk.check(pk.pkm_forward(h, q, C, V, B, H, n, k, out, idx, w), "forward")
            pk.check(pk.pkm_backward(h, q, C, V, B, H, n, k, idx, w, dout, dq, dC, dVt),
                     "backward")
            pk.check(pk.pkm_backward_sparse(h, q, C, V, B, H, n, k, idx, w, dout, dq, dC, rows,
                                            grad, nr), "backward_sparse")
            pk.check(pk.pkm_forward_host(h, qh, C, V, B, H, n, k, oh), "forward_host")
            pk.check(pk.pkm_forward_host_async(h, qh, C, V, B, H, n, k, oh, ev), "async")
            ev.synchronize()
            torch.cuda.synchronize()

        round_of_calls()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(3):
            round_of_calls()
        assert torch.cuda.mem_get_info()[0] == free0
        assert pk.pkm_get_status(h) == pk.PKM_OK
    finally:
        pk.pkm_destroy(h)
