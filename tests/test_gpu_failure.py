"""Failure reporting on the GPU without a fault: a bounded wait that runs out.

PKM_OPT_TEST_STALL (bit 0) holds back the selection kernel's loads, so the
MMA warp's wait for its first stage runs out (about 2 s); bit 1 makes the
bulk-copy value read issue no copy, so its consumers' first waits run out.
The kernel records PKM_ERR_TIMEOUT in the status word and every warp returns;
the tests then check that the status is reported once and that the same
context computes correct results afterwards.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_lookup, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")


@pytest.mark.parametrize("form", [1, 2])
def test_bounded_wait_runs_out_is_reported_and_context_stays_usable(form):
    # form 1: the one-SM selection kernel; form 2: the two-SM one, whose two
    # CTAs both run out (each on its own waits) and meet at the final cluster
    # barrier
    B, H, d_q, n, d_v, k = 256, 1, 128, 256, 64, 16
    s = synth.seed_of(dict(cfg_id=160))
    q = synth.normal(s, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(s, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    h = pk.pkm_create(pk.make_config(d_q, d_v, B, H, n, k, q_dtype=pk.PKM_BF16))
    try:
        tq, tC = to_device(q, "bf16"), to_device(C, "bf16")
        idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w = torch.empty(B, H, k, device="cuda")
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_SELECT_FORM, form), "set_option")
        assert pk.pkm_set_option(h, pk.PKM_OPT_TEST_STALL, 4) == pk.PKM_ERR_OPTION
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_TEST_STALL, 1), "set_option")
        pk.check(pk.pkm_lookup(h, tq, tC, B, H, n, k, idx, w), "pkm_lookup")
        assert pk.pkm_get_status(h) == pk.PKM_ERR_TIMEOUT
        assert pk.pkm_get_status(h) == pk.PKM_OK  # reported once, then cleared
        # the same context, the stall off: exact results again
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_TEST_STALL, 0), "set_option")
        pk.check(pk.pkm_lookup(h, tq, tC, B, H, n, k, idx, w), "pkm_lookup")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        ref = oracle.lookup(q, C, B, H, d_q, n, k)
        res = compare_lookup(idx.cpu().numpy(), w.cpu().numpy(), ref, q, C, "bf16", H, d_q, n)
        assert res["failures"] == 0 and res["w_ok"], res
    finally:
        pk.pkm_destroy(h)
    torch.cuda.synchronize()


def test_read_bounded_wait_runs_out_is_reported_and_context_stays_usable():
    B, H, n, d_v, k = 64, 2, 16, 512, 8   # 1 KB rows: the bulk-copy read
    N = n * n
    rng = np.random.default_rng(5)
    idx_np = rng.integers(0, N, (B, H, k)).astype(np.int64)
    w_np = rng.uniform(0.1, 1.0, (B, H, k)).astype(np.float32)
    V = synth.normal(161, 3, N * d_v, 1.0, dtype="bf16")
    h = pk.pkm_create(pk.make_config(32, d_v, B, H, n, k, q_dtype=pk.PKM_BF16))
    try:
        dV = to_device(V, "bf16")
        idx, w = torch.from_numpy(idx_np).cuda(), torch.from_numpy(w_np).cuda()
        out = torch.empty(B, d_v, device="cuda")
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_TEST_STALL, 2), "set_option")
        pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out), "pkm_gather")
        assert pk.pkm_get_status(h) == pk.PKM_ERR_TIMEOUT
        assert pk.pkm_get_status(h) == pk.PKM_OK
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_TEST_STALL, 0), "set_option")
        pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out), "pkm_gather")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        ref = oracle.gather(V, N, d_v, idx_np, w_np.astype(np.float64))
        err = np.abs(out.cpu().numpy().astype(np.float64) - ref) / (1 + np.abs(ref))
        assert err.max() <= 1e-5, float(err.max())
    finally:
        pk.pkm_destroy(h)
    torch.cuda.synchronize()
