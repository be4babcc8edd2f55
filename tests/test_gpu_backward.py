"""Parity of the backward pass (pkm_backward) with the fp64 oracle.

The selection is fixed (the top-k choices carry no gradient), so the inputs
are the forward's q, subkeys, values, a selection (idx, w) and the gradient
dout at the read's output.  In the small cases idx and w come from the
oracle's own lookup; at the full page sizes from the seeded stand-in
selection of synth.selections.  Tolerances are bounds derived from the
kernels' arithmetic (see gpu_error_bounds); dq is overwritten, dsubkeys and
dvalues are added to, which the tests check with non-zero starting values.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import to_device, widen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")

U = 2.0 ** -24          # fp32 unit roundoff
DC0, DV0 = 0.5, 0.25    # starting values of the accumulated gradients (exact in fp32)


def gpu_error_bounds(q64, C64, Vsel, idx, w, dout, dw, n, k, B_gemm):
    """Per-element bounds on |gpu - exact| for dq [B,H,d_q] and for the
    dsubkeys contributions of these queries [H,2,n,d_q/2].

    Arithmetic of the GPU path: dw is a per-lane fp32 fma chain of d_v/32
    terms plus 5 shuffle additions; ds_j = w_j (dw_j - sum_l w_l dw_l) in
    fp32; the per-subkey sums DS are fp32 sums of at most k terms; dq sums
    at most k fp32 fused multiply-adds DS * C per element (one per distinct
    winning subkey) and dC at most B of DS * q (one per query that selected
    the subkey), each product of an fp32 DS and a bf16 operand exact inside
    its fma.
    """
    B, H, _ = idx.shape
    d_q = q64.shape[-1]
    hd = d_q // 2
    d_v = dout.shape[1]
    A = np.einsum("bc,bhjc->bhj", np.abs(dout), np.abs(Vsel))
    edw = (d_v / 32 + 6) * U * A
    sw_err = (w * edw).sum(-1, keepdims=True) + 6 * U * (w * np.abs(dw)).sum(-1, keepdims=True)
    ds = w * (dw - (w * dw).sum(-1, keepdims=True))
    eds = w * (edw + sw_err) + 3 * U * np.abs(ds)
    DSabs = np.zeros((H, 2, B, n))
    EDS = np.zeros((H, 2, B, n))
    bb = np.broadcast_to(np.arange(B)[:, None], (B, k))
    for h in range(H):
        for half, a in enumerate((idx[:, h] // n, idx[:, h] % n)):
            np.add.at(DSabs[h, half], (bb, a), np.abs(ds[:, h]))
            np.add.at(EDS[h, half], (bb, a), eds[:, h])
    EDS += k * U * DSabs
    tol_dq = np.empty((B, H, d_q))
    tol_dC = np.empty((H, 2, n, hd))
    for h in range(H):
        for half in range(2):
            Cabs = np.abs(C64[h, half])
            qabs = np.abs(q64[:, h, half * hd:(half + 1) * hd])
            tol_dq[:, h, half * hd:(half + 1) * hd] = (
                EDS[h, half] @ Cabs + (k + 2) * U * (DSabs[h, half] @ Cabs))
            tol_dC[h, half] = (EDS[h, half].T @ qabs +
                               (B_gemm + 2) * U * (DSabs[h, half].T @ qabs))
    return tol_dq, tol_dC, ds


def dvalue_bound(idx, w, dout, rows):
    """|gpu - exact| bound for dvalues rows of m selections: fused multiply-adds
    of w * dout into fp32 partial sums of up to 4 selections, each added onto
    the row (at most 2m + 1 roundings, in any order)."""
    slot = {int(r): i for i, r in enumerate(rows)}
    absum = np.zeros((len(rows), dout.shape[1]))
    mult = np.zeros(len(rows))
    B = idx.shape[0]
    for b in range(B):
        for r, wt in zip(idx[b].ravel(), w[b].ravel()):
            i = slot.get(int(r))
            if i is not None:
                absum[i] += abs(wt) * np.abs(dout[b])
                mult[i] += 1
    return (2 * mult[:, None] + 2) * U * (absum + DV0)


def run_backward(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout, max_B=None, split=False):
    """pkm_backward through the C ABI (or, split, pkm_backward_read then
    pkm_backward_scores); returns (dq, dC - DC0, dV tensor, status[, dw])."""
    cfg = pk.make_config(d_q, d_v, max_B or max(B, 1), H, n, k, q_dtype=pk.PKM_BF16,
                         value_dtype=pk.PKM_F32 if vdt == "f32" else pk.PKM_BF16,
                         with_backward=1)
    h = pk.pkm_create(cfg)
    try:
        tq, tC = to_device(q, "bf16"), to_device(C, "bf16")
        tV = to_device(V, vdt)
        tidx = torch.from_numpy(np.ascontiguousarray(idx, np.int64)).cuda()
        tw = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
        tdout = torch.from_numpy(np.ascontiguousarray(dout, np.float32)).cuda()
        dq = torch.full((max(B, 1), H, d_q), float("nan"), device="cuda")
        dC = torch.full((H, 2, n, d_q // 2), DC0, device="cuda")
        dV = torch.full((n * n, d_v), DV0, device="cuda")
        if split:
            dw = torch.full((max(B, 1), H, k), float("nan"), device="cuda")
            pk.check(pk.pkm_backward_read(h, tV, B, H, n, k, tidx, tw, tdout, dw, dV),
                     "pkm_backward_read")
            pk.check(pk.pkm_backward_scores(h, tq, tC, B, H, n, k, tidx, tw, dw, dq, dC),
                     "pkm_backward_scores")
        else:
            pk.check(pk.pkm_backward(h, tq, tC, tV, B, H, n, k, tidx, tw, tdout, dq, dC, dV),
                     "pkm_backward")
        status = pk.pkm_get_status(h)
        res = dq.cpu().numpy()[:B], (dC - DC0).cpu().numpy(), dV, status
        return res + (dw.cpu().numpy()[:B],) if split else res
    finally:
        pk.pkm_destroy(h)


def check_against_oracle(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout, got):
    gdq, gdC, gdV, status = got
    assert status == pk.PKM_OK
    q64 = widen(q, "bf16").reshape(B, H, d_q)
    C64 = widen(C, "bf16").reshape(H, 2, n, d_q // 2)
    V2 = V.reshape(n * n, d_v)
    rows = np.unique(idx)
    ref = oracle.backward(q, C, V, B, H, d_q, n, d_v, k, idx, w.astype(np.float64), dout,
                          dvalue_rows=rows)
    Vsel = widen(V2[idx.ravel()], vdt).reshape(B, H, k, d_v)
    w64 = w.astype(np.float64)
    tol_dq, tol_dC, ds = gpu_error_bounds(q64, C64, Vsel, idx, w64, dout.astype(np.float64),
                                          ref["dw"], n, k, B)
    err = np.abs(gdq - ref["dq"])
    assert (err <= tol_dq).all(), float((err / np.maximum(tol_dq, 1e-300)).max())
    err = np.abs(gdC - ref["dsubkeys"])
    assert (err <= tol_dC + U * (DC0 + np.abs(ref["dsubkeys"]))).all()
    # the bound is tight enough to see a wrong operand, a dropped term or a
    # low-precision rounding of the score gradients (bf16 would be 2^-9 of
    # |dq|): a thousandth of |dq| at most for most sizable entries
    big = np.abs(ref["dq"]) > 1e-3 * np.abs(ref["dq"]).max()
    if big.any():
        assert np.median(tol_dq[big] / np.abs(ref["dq"][big])) < 1e-3
    gV = gdV[torch.from_numpy(rows).cuda()].cpu().numpy()
    err = np.abs(gV - (DV0 + ref["dvalues"]))
    assert (err <= dvalue_bound(idx, w64, dout, rows)).all()
    # rows no query selected keep their starting value exactly
    mask = torch.ones(n * n, dtype=torch.bool, device="cuda")
    mask[torch.from_numpy(rows).cuda()] = False
    assert bool((gdV[mask] == DV0).all())
    return ref


def lookup_case(seed, B, H, d_q, n, d_v, k, vdt="bf16"):
    """Inputs from the seeded generator; the selection from the oracle's lookup."""
    s = synth.seed_of(dict(cfg_id=100 + seed))
    q = synth.normal(s, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(s, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    V = synth.normal(s, 3, n * n * d_v, 1.0 / d_v, dtype=vdt)
    dout = synth.normal(s, 15, B * d_v, 1.0).reshape(B, d_v).astype(np.float64)
    ref = oracle.lookup(q, C, B, H, d_q, n, k)
    return q, C, V, ref["idx"], ref["w"].astype(np.float32), dout


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, d_v, k, values
    (300, 2, 128, 64, 256, 16, "bf16"),     # ragged batch, two heads
    (130, 3, 64, 33, 64, 8, "f32"),         # odd n_keys (unpaired bf16 stores), fp32 table
    (64, 1, 1024, 1024, 1024, 32, "bf16"),  # the page's d, n_keys and k
    (1, 4, 32, 100, 32, 7, "bf16"),          # one query, odd k, small d_q, n_keys not 2^p
    (257, 1, 16, 40, 16, 1, "f32"),          # k = 1, the smallest d_q and d_v
])
def test_backward_matches_oracle(shape):
    B, H, d_q, n, d_v, k, vdt = shape
    q, C, V, idx, w, dout = lookup_case(sum(shape[:6]), B, H, d_q, n, d_v, k, vdt)
    got = run_backward(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout)
    check_against_oracle(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout, got)


def test_backward_split_calls():
    # the two halves through their own entry points; dw is the oracle's
    # within the fp32 dot-product bound
    B, H, d_q, n, d_v, k = 200, 2, 128, 64, 512, 16
    q, C, V, idx, w, dout = lookup_case(3, B, H, d_q, n, d_v, k)
    got = run_backward(q, C, V, "bf16", B, H, d_q, n, d_v, k, idx, w, dout, split=True)
    ref = check_against_oracle(q, C, V, "bf16", B, H, d_q, n, d_v, k, idx, w, dout, got[:4])
    Vsel = widen(V.reshape(n * n, d_v)[idx.ravel()], "bf16").reshape(B, H, k, d_v)
    A = np.einsum("bc,bhjc->bhj", np.abs(dout), np.abs(Vsel))
    assert (np.abs(got[4] - ref["dw"]) <= (d_v / 32 + 6) * U * A).all()


@pytest.mark.parametrize("vdt", ["bf16", "f32"])
def test_backward_concentrated_selection(vdt):
    # usage collapse ("Keeping the memory in use"): 9,600 selections on 300
    # rows of a 4,096-row table, so one 256-row bucket holds more than one
    # chunk of selections (rows shared between CTAs, vector atomic adds) and
    # most rows more than one piece; plus one row every query selects
    B, H, d_q, n, d_v, k = 300, 2, 64, 64, 128, 16
    s = synth.seed_of(dict(cfg_id=140))
    q = synth.normal(s, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(s, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    V = synth.normal(s, 3, n * n * d_v, 1.0 / d_v, dtype=vdt)
    dout = synth.normal(s, 15, B * d_v, 1.0).reshape(B, d_v).astype(np.float64)
    u = synth.uniform(s, 12, B * H * k).reshape(B, H, k)
    idx = np.minimum((u * 300).astype(np.int64), 299)
    idx[:, 0, 0] = 4000  # a hot row in another bucket
    e = -np.log1p(-synth.uniform(s, 14, B * H * k)).reshape(B, H, k)
    w = (e / e.sum(-1, keepdims=True)).astype(np.float32)
    got = run_backward(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout)
    check_against_oracle(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout, got)


def run_backward_sparse(q, C, V, vdt, B, H, d_q, n, d_v, k, idx, w, dout):
    """pkm_backward_sparse; returns (dq, dC, rows, grad_rows, status)."""
    cfg = pk.make_config(d_q, d_v, B, H, n, k, q_dtype=pk.PKM_BF16,
                         value_dtype=pk.PKM_F32 if vdt == "f32" else pk.PKM_BF16,
                         with_backward=1)
    h = pk.pkm_create(cfg)
    try:
        E = B * H * k
        tq, tC, tV = to_device(q, "bf16"), to_device(C, "bf16"), to_device(V, vdt)
        tidx = torch.from_numpy(np.ascontiguousarray(idx, np.int64)).cuda()
        tw = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
        tdout = torch.from_numpy(np.ascontiguousarray(dout, np.float32)).cuda()
        dq = torch.full((B, H, d_q), float("nan"), device="cuda")
        dC = torch.zeros(H, 2, n, d_q // 2, device="cuda")
        rows = torch.full((E,), -7, dtype=torch.int64, device="cuda")
        grad = torch.full((E, d_v), float("nan"), device="cuda")
        nr = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        pk.check(pk.pkm_backward_sparse(h, tq, tC, tV, B, H, n, k, tidx, tw, tdout, dq, dC, rows,
                                        grad, nr), "pkm_backward_sparse")
        status = pk.pkm_get_status(h)
        m = int(nr.item())
        return (dq.cpu().numpy(), dC.cpu().numpy(), rows[:m].cpu().numpy(),
                grad[:m].cpu().numpy(), status)
    finally:
        pk.pkm_destroy(h)


def concentrated_case(vdt):
    B, H, d_q, n, d_v, k = 300, 2, 64, 64, 128, 16
    s = synth.seed_of(dict(cfg_id=140))
    q = synth.normal(s, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(s, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    V = synth.normal(s, 3, n * n * d_v, 1.0 / d_v, dtype=vdt)
    dout = synth.normal(s, 15, B * d_v, 1.0).reshape(B, d_v).astype(np.float64)
    u = synth.uniform(s, 12, B * H * k).reshape(B, H, k)
    idx = np.minimum((u * 300).astype(np.int64), 299)
    idx[:, 0, 0] = 4000
    e = -np.log1p(-synth.uniform(s, 14, B * H * k)).reshape(B, H, k)
    w = (e / e.sum(-1, keepdims=True)).astype(np.float32)
    return (B, H, d_q, n, d_v, k), q, C, V, idx, w, dout


@pytest.mark.parametrize("case", ["lookup", "concentrated_bf16", "concentrated_f32", "bad_index"])
def test_backward_sparse_matches_oracle(case):
    # the sparse value-table gradient: the distinct selected rows (ascending,
    # exact) and their gradients (fp32 bound); dq and dsubkeys as the dense form
    if case.startswith("concentrated"):
        vdt = case.split("_")[1]
        (B, H, d_q, n, d_v, k), q, C, V, idx, w, dout = concentrated_case(vdt)
    else:
        vdt = "bf16"
        B, H, d_q, n, d_v, k = 200, 2, 128, 64, 256, 16
        q, C, V, idx, w, dout = lookup_case(21, B, H, d_q, n, d_v, k)
    gidx = idx.copy()
    if case == "bad_index":
        gidx[3, 1, 5] = -1  # left out of the rows, recorded in the status
    gdq, gdC, rows, grad, status = run_backward_sparse(q, C, V, vdt, B, H, d_q, n, d_v, k, gidx, w,
                                                       dout)
    assert status == (pk.PKM_ERR_BAD_INDEX if case == "bad_index" else pk.PKM_OK)
    valid = gidx[gidx >= 0]
    want_rows = np.unique(valid)
    assert np.array_equal(rows, want_rows)
    if case == "bad_index":
        return
    ref = oracle.backward(q, C, V, B, H, d_q, n, d_v, k, idx, w.astype(np.float64), dout,
                          dvalue_rows=rows)
    w64 = w.astype(np.float64)
    # (the bound counts a starting value DV0 the sparse rows do not have: looser by that term)
    assert (np.abs(grad - ref["dvalues"]) <= dvalue_bound(idx, w64, dout, rows)).all()
    q64 = widen(q, "bf16").reshape(B, H, d_q)
    C64 = widen(C, "bf16").reshape(H, 2, n, d_q // 2)
    Vsel = widen(V.reshape(n * n, d_v)[idx.ravel()], vdt).reshape(B, H, k, d_v)
    tol_dq, tol_dC, _ = gpu_error_bounds(q64, C64, Vsel, idx, w64, dout, ref["dw"], n, k, B)
    assert (np.abs(gdq - ref["dq"]) <= tol_dq).all()
    assert (np.abs(gdC - ref["dsubkeys"]) <= tol_dC).all()


def test_backward_single_winner_closed_form():
    # k = 1: w = 1, so ds = 0: dq is exactly 0, dsubkeys unchanged, and
    # dvalues[idx] gains the dout of every query that selected it
    B, H, d_q, n, d_v, k = 40, 2, 64, 16, 128, 1
    q, C, V, idx, w, dout = lookup_case(7, B, H, d_q, n, d_v, k)
    assert (w == 1).all()
    gdq, gdC, gdV, status = run_backward(q, C, V, "bf16", B, H, d_q, n, d_v, k, idx, w, dout)
    assert status == pk.PKM_OK
    assert (gdq == 0).all() and (gdC == 0).all()
    want = np.full((n * n, d_v), DV0)
    for b in range(B):
        for h in range(H):
            want[idx[b, h, 0]] += dout[b]
    rows = np.unique(idx)
    got = gdV.cpu().numpy()
    assert (np.abs(got[rows] - want[rows]) <= dvalue_bound(idx, w, dout, rows)).all()
    untouched = np.setdiff1d(np.arange(n * n), rows)
    assert (got[untouched] == DV0).all()


def test_backward_empty_batch_and_unarmed_handle():
    d_q, n, d_v, k, H = 64, 16, 64, 4, 1
    cfg = pk.make_config(d_q, d_v, 8, H, n, k, q_dtype=pk.PKM_BF16, with_backward=1)
    h = pk.pkm_create(cfg)
    try:
        buf = torch.zeros(1 << 16, device="cuda")
        assert pk.pkm_backward(h, buf, buf, buf, 0, H, n, k, buf, buf, buf, buf, buf, buf) \
            == pk.PKM_OK
        assert pk.pkm_backward(h, buf, buf, buf, 9, H, n, k, buf, buf, buf, buf, buf, buf) \
            == pk.PKM_ERR_RANGE
        assert pk.pkm_backward(h, buf, buf, buf, 1, H, n, k, buf, buf, buf, buf, buf, None) \
            == pk.PKM_ERR_INVALID
        assert pk.pkm_get_status(h) == pk.PKM_OK
    finally:
        pk.pkm_destroy(h)
    h = pk.pkm_create(pk.make_config(d_q, d_v, 8, H, n, k, q_dtype=pk.PKM_BF16))
    try:
        buf = torch.zeros(1 << 16, device="cuda")
        assert pk.pkm_backward(h, buf, buf, buf, 1, H, n, k, buf, buf, buf, buf, buf, buf) \
            == pk.PKM_ERR_NO_BACKWARD
    finally:
        pk.pkm_destroy(h)


def test_backward_bad_index_recorded():
    # an index outside the table is reported and contributes nothing; the
    # other queries' gradients are unaffected
    B, H, d_q, n, d_v, k = 24, 1, 64, 16, 64, 4
    q, C, V, idx, w, dout = lookup_case(11, B, H, d_q, n, d_v, k)
    bad = idx.copy()
    bad[0, 0, 2] = n * n
    gdq, _, gdV, status = run_backward(q, C, V, "bf16", B, H, d_q, n, d_v, k, bad, w, dout)
    assert status == pk.PKM_ERR_BAD_INDEX
    assert np.isfinite(gdq).all() and bool(torch.isfinite(gdV).all())
    ref = oracle.backward(q[H * d_q:], C, V, B - 1, H, d_q, n, d_v, k, idx[1:],
                          w[1:].astype(np.float64), dout[1:], dvalue_rows=[0])
    q64 = widen(q, "bf16").reshape(B, H, d_q)[1:]
    C64 = widen(C, "bf16").reshape(H, 2, n, d_q // 2)
    Vsel = widen(V.reshape(n * n, d_v)[idx[1:].ravel()], "bf16").reshape(B - 1, H, k, d_v)
    tol_dq, _, _ = gpu_error_bounds(q64, C64, Vsel, idx[1:], w[1:].astype(np.float64), dout[1:],
                                    ref["dw"], n, k, B)
    assert (np.abs(gdq[1:] - ref["dq"]) <= tol_dq).all()


@pytest.mark.slow
def test_backward_page_sizes_sampled():
    """The training-step workload's shapes and the benchmark's handle configuration;
    the oracle recomputes sampled dq rows (one query each), dsubkeys rows
    (the queries that selected that subkey) and dvalues rows (the queries
    that selected that row)."""
    c = synth.CONFIGS["page_train"]
    B, H, d_q, n, d_v, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "d_v", "k"))
    q, C, V = synth.queries(c), synth.subkeys(c), synth.values(c)
    a1, a2, w = synth.selections(c)
    idx = a1 * n + a2
    dout = synth.output_grads(c).astype(np.float64)
    gdq, gdC, gdV, status = run_backward(q, C, V, "bf16", B, H, d_q, n, d_v, k, idx, w, dout)
    assert status == pk.PKM_OK
    q3 = q.reshape(B, H * d_q)
    C64 = widen(C, "bf16").reshape(H, 2, n, d_q // 2)
    V2 = V.reshape(n * n, d_v)

    def sub(bs, rows=None):
        bs = np.asarray(bs)
        r = oracle.backward(q3[bs], C, V, len(bs), H, d_q, n, d_v, k, idx[bs],
                            w[bs].astype(np.float64), dout[bs],
                            dvalue_rows=[] if rows is None else rows)
        Vsel = widen(V2[idx[bs].ravel()], "bf16").reshape(len(bs), H, k, d_v)
        q64 = widen(q3[bs], "bf16").reshape(len(bs), H, d_q)
        tq, tC, _ = gpu_error_bounds(q64, C64, Vsel, idx[bs], w[bs].astype(np.float64),
                                     dout[bs], r["dw"], n, k, B)
        return r, tq, tC

    rng = np.random.default_rng(5)
    qs = np.unique(np.concatenate([[0, B - 1], rng.integers(0, B, 14)]))
    for b in qs:
        r, tq, _ = sub([b])
        assert (np.abs(gdq[b] - r["dq"][0]) <= tq[0]).all(), b
    for h, half in [(0, 0), (H - 1, 1), (1, 1)]:
        sk = (idx[:, h] // n if half == 0 else idx[:, h] % n)
        a = int(sk[rng.integers(0, B), rng.integers(0, k)])
        bs = np.nonzero((sk == a).any(-1))[0]
        r, _, tC = sub(bs)
        err = np.abs(gdC[h, half, a] - r["dsubkeys"][h, half, a])
        assert (err <= tC[h, half, a] + U * (DC0 + np.abs(r["dsubkeys"][h, half, a]))).all()
    for _ in range(3):
        row = int(idx[rng.integers(0, B), rng.integers(0, H), rng.integers(0, k)])
        bs = np.nonzero((idx == row).any(-1).any(-1))[0]
        r, _, _ = sub(bs, rows=[row])
        gV = gdV[row].cpu().numpy()
        bound = dvalue_bound(idx[bs], w[bs].astype(np.float64), dout[bs], [row])[0]
        assert (np.abs(gV - (DV0 + r["dvalues"][0])) <= bound).all()
