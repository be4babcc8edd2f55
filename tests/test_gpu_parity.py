"""GPU parity against the fp64 oracle, through the C ABI.

Workloads small enough for the oracle to check every output: the fp32 tiny
problem (CUDA-core path), the bf16 mid problem (tensor-core path), and edge
shapes: ragged batch tails, n_keys not a multiple of the chunk width, k = 1,
k = n_keys, exact integer ties, B = 0, out-of-range indices.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, compare_lookup, compare_out, make_handle, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")


def run_forward(cfgd, q, C, V, B=None, hint_z=None, report=None, form=None):
    B = cfgd["B"] if B is None else B
    H, k, d_v = cfgd["H"], cfgd["k"], cfgd["d_v"]
    h, _ = make_handle(dict(cfgd, B=max(B, 1)))
    try:
        if hint_z is not None:
            pk.check(pk.pkm_set_option(h, pk.PKM_OPT_HINT_Z, hint_z), "set_option")
        if form is not None:
            pk.check(pk.pkm_set_option(h, pk.PKM_OPT_SELECT_FORM, form), "set_option")
        dq, dC, dV = (to_device(x, cfgd["dtype"]) for x in (q, C, V))
        out = torch.empty(B, d_v, device="cuda")
        idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w = torch.empty(B, H, k, device="cuda")
        pk.check(pk.pkm_forward(h, dq, dC, dV, B, H, cfgd["n_keys"], k, out, idx, w), "forward")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        if report is not None and cfgd["dtype"] == "bf16":
            report["fallback"] = pk.pkm_get_fallback_count(h)
        return out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    finally:
        pk.pkm_destroy(h)


def check_against_oracle(cfgd, q, C, V, max_near_frac=0.01, hint_z=None, report=None,
                         form=None):
    B, H, d_q, n, d_v, k = (cfgd[x] for x in ("B", "H", "d_q", "n_keys", "d_v", "k"))
    out, idx, w = run_forward(cfgd, q, C, V, hint_z=hint_z, report=report, form=form)
    ref = oracle.lookup(q, C, B, H, d_q, n, k)
    rep = compare_lookup(idx, w, ref, q, C, cfgd["dtype"], H, d_q, n)
    assert rep["failures"] == 0, rep
    assert rep["near_ties"] <= max_near_frac * B * H, rep
    assert rep["w_ok"], rep
    ref_out = oracle.gather(V, n * n, d_v, ref["idx"], ref["w"])
    err = compare_out(out, V, n * n, d_v, idx, ref["idx"], ref["w"], ref_out)
    assert err <= TOL, err
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-5)
    return rep


def cfg_inputs(name):
    c = synth.CONFIGS[name]
    return c, synth.queries(c), synth.subkeys(c), synth.values(c)


def test_tiny_fp32_matches_oracle_and_brute_force():
    c, q, C, V = cfg_inputs("tiny")
    check_against_oracle(c, q, C, V)
    _, idx, _ = run_forward(c, q, C, V)
    bi, _ = oracle.brute_topk(q, C, c["B"], c["H"], c["d_q"], c["n_keys"], c["k"])
    assert (idx == bi).all(-1).mean() > 0.99


def test_mid_bf16_matches_oracle():
    c, q, C, V = cfg_inputs("mid")
    info = {}
    rep = check_against_oracle(c, q, C, V, report=info)
    print("mid parity:", rep, info)
    # normally distributed scores: the automatic threshold hint never falls back
    assert info["fallback"] == 0


def random_case(seed, B, H, d_q, n, d_v, k, dtype="bf16", kvar=None):
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=d_v, k=k, dtype=dtype)
    kvar = kvar if kvar is not None else 2.0 / d_q
    q = synth.normal(seed, 1, B * H * d_q, 1.0, dtype=dtype)
    C = synth.normal(seed, 2, H * 2 * n * (d_q // 2), kvar, dtype=dtype)
    V = synth.normal(seed, 3, n * n * d_v, 1.0 / d_v, dtype=dtype)
    return c, q, C, V


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, d_v, k
    (300, 2, 128, 256, 128, 16),    # ragged batch tail (300 = 2*128 + 44)
    (130, 3, 192, 100, 64, 8),      # n_keys not a multiple of 32, d_q/2 not a multiple of 64
    (257, 1, 64, 520, 256, 32),     # three chunks, the last one partial
    (64, 2, 256, 48, 128, 1),       # k = 1: argmax per half
    (40, 1, 32, 20, 64, 20),        # k = n_keys: every key is a candidate
    (129, 2, 1024, 1024, 1024, 32),  # page-width rows, small batch
    (64, 8, 256, 256, 128, 32),     # eight heads (the skewed workload's H)
    (70, 1, 128, 2048, 64, 32),     # 16 chunks per half (the large workload's n_keys)
    (130, 2, 2048, 256, 128, 32),   # 16 k-slabs per chunk: one epilogue set, 5 tile stages
    (200, 1, 1152, 300, 64, 16),    # 9 k-slabs (the narrowest one-set shape), ragged chunks
])
def test_bf16_shapes(shape):
    c, q, C, V = random_case(sum(shape), *shape)
    check_against_oracle(c, q, C, V)


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, d_v, k: the two-SM selection form forced
    (100, 1, 128, 256, 64, 16),     # one pair tile: the second CTA's rows all out of range
    (300, 2, 128, 256, 128, 16),    # second pair tile ragged (300 = 256 + 44)
    (257, 1, 64, 520, 256, 32),     # three 256-key chunks, the last one holding 8 keys
    (130, 3, 192, 100, 64, 8),      # n below one CTA's 128-key half; 3 k-slabs, the last partial
    (64, 2, 256, 48, 128, 1),       # k = 1
    (40, 1, 32, 20, 64, 20),        # k = n_keys, one k-slab of 16 columns
    (520, 2, 1024, 1024, 1024, 32),  # page-width rows: 4 chunks of 8 k-slabs
    (300, 8, 256, 256, 128, 32),    # eight heads
    (129, 1, 128, 2048, 64, 32),    # 8 chunks per half (the large workload's n_keys)
    (260, 2, 2048, 512, 128, 32),   # 16 k-slabs per chunk (the large workload's width)
])
@pytest.mark.parametrize("form", [2, 3])
def test_two_sm_form_shapes(shape, form):
    c, q, C, V = random_case(sum(shape) + 5, *shape)
    check_against_oracle(c, q, C, V, form=form)


@pytest.mark.parametrize("form", [2, 3])
@pytest.mark.parametrize("z", [1e30, 1.53, -1e30])
def test_two_sm_form_exact_for_any_threshold_hint(z, form):
    # every row retried (huge z: the lists are marked and the retry pass
    # selects their 128-row units with the one-SM kernel), about half of them,
    # or none with every score logged (repeated compactions from both log ends)
    c, q, C, V = random_case(99, 520, 2, 256, 1024, 128, 32)
    info = {}
    check_against_oracle(c, q, C, V, hint_z=z, report=info, form=form)
    if z == 1e30:
        assert info["fallback"] == c["B"] * c["H"]
    if z < 0:
        assert info["fallback"] == 0


@pytest.mark.parametrize("form", [1, 2, 3])
def test_forms_agree_bit_for_bit(form):
    # the mid workload through each selection form gives the same indices,
    # weights and outputs as the automatic choice
    c, q, C, V = cfg_inputs("mid")
    want = run_forward(c, q, C, V)
    got = run_forward(c, q, C, V, form=form)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, d_v, k: bf16 lookups with 32 < k <= 64 run on the CUDA cores
    (70, 2, 128, 256, 128, 48),     # ragged batch, k^2 = 2304 candidates
    (33, 1, 64, 100, 64, 64),       # k = 64 of 100 subkeys per half
    (20, 4, 1024, 1024, 1024, 40),  # page-width rows
])
def test_bf16_large_k(shape):
    c, q, C, V = random_case(sum(shape) + 1, *shape)
    check_against_oracle(c, q, C, V)


def test_bf16_large_k_exact_ties():
    # integer-valued bf16 inputs: exact fp32 scores, so the CUDA-core path's
    # tie orders must reproduce the oracle's bit for bit at k = 40
    rng = np.random.default_rng(8)
    B, H, d_q, n, d_v, k = 50, 2, 64, 64, 32, 40
    qf = rng.integers(-3, 4, (B, H, d_q)).astype(np.float32)
    Cf = rng.integers(-2, 3, (H, 2, n, d_q // 2)).astype(np.float32)
    Cf[:, 0, 10:20] = Cf[:, 0, 0:10]
    Vf = rng.standard_normal((n * n, d_v)).astype(np.float32)
    q, C, V = synth.f32_to_bf16(qf), synth.f32_to_bf16(Cf), synth.f32_to_bf16(Vf)
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=d_v, k=k, dtype="bf16")
    out, idx, w = run_forward(c, q.ravel(), C.ravel(), V.ravel())
    ref = oracle.lookup(q.ravel(), C.ravel(), B, H, d_q, n, k)
    assert np.array_equal(idx, ref["idx"])
    assert (np.abs(w - ref["w"]) <= 1e-6 * (1 + ref["w"])).all()


@pytest.mark.parametrize("z", [1e30, -1e30, -1.0, 0.5, 1.53, 2.5])
def test_selection_exact_for_any_threshold_hint(z):
    # The per-row threshold hint only steers cost.  A huge z leaves every row
    # with too few logged scores, so every row tile goes through the retry
    # pass (selected again without the hint); z = 1.53 puts about KL of the
    # 512 scores above the hint, so about half the rows miss and retried and
    # untouched units mix; a very negative z logs every score and exercises
    # repeated log compactions.  Either way the result is the oracle's.
    c, q, C, V = random_case(99, 260, 2, 256, 512, 128, 32)
    info = {}
    check_against_oracle(c, q, C, V, hint_z=z, report=info)
    if z == 1e30:
        assert info["fallback"] == c["B"] * c["H"]
    if z <= -1.0:
        assert info["fallback"] == 0


@pytest.mark.parametrize("z", [1e30, 1.53, -1e30])
def test_one_set_selection_exact_for_any_threshold_hint(z):
    # the one-set form (wide half-queries) with every row retried (huge z),
    # about half of them (z = 1.53), or none and every score logged
    c, q, C, V = random_case(77, 260, 2, 2048, 512, 128, 32)
    info = {}
    check_against_oracle(c, q, C, V, hint_z=z, report=info)
    if z == 1e30:
        assert info["fallback"] == c["B"] * c["H"]
    if z < 0:
        assert info["fallback"] == 0


@pytest.mark.parametrize("z", [1e30, 1.86])
def test_short_lists_exact_for_any_threshold_hint(z):
    # k <= 16 (16-entry per-half lists, the merge's KL = 16 form) with every
    # row retried (huge z) or about half of them (z = 1.86 puts about 16 of
    # the 512 scores above the hint), on a batch that ends inside a row tile
    # (200 = 128 + 72: the retry pass's two CTAs of the last unit, one partly
    # and one wholly past the batch)
    c, q, C, V = random_case(123, 200, 3, 256, 512, 64, 12)
    info = {}
    check_against_oracle(c, q, C, V, hint_z=z, report=info)
    if z == 1e30:
        assert info["fallback"] == c["B"] * c["H"]


def test_fp32_shapes():
    c, q, C, V = random_case(7, 33, 3, 48, 40, 32, 12, dtype="f32", kvar=1.0)
    check_against_oracle(c, q, C, V)


@pytest.mark.parametrize("dtype,form", [("bf16", 1), ("bf16", 2), ("f32", None)])
def test_exact_integer_ties_bit_exact(dtype, form):
    # Small integers are exact in bf16/fp32 and every partial sum stays exact
    # in fp32, so GPU and oracle scores are identical: the tie rule (lower
    # subkey index per half, lower flat index overall) must match bit for bit.
    rng = np.random.default_rng(3)
    B, H, d_q, n, d_v, k = 200, 2, 64, 64, 32, 16
    qf = rng.integers(-3, 4, (B, H, d_q)).astype(np.float32)
    Cf = rng.integers(-2, 3, (H, 2, n, d_q // 2)).astype(np.float32)
    Cf[:, 0, 10:20] = Cf[:, 0, 0:10]   # duplicated rows force exact ties in half 1
    Cf[:, 1, 40:60] = Cf[:, 1, 5][:, None, :]  # and many in half 2
    Vf = rng.standard_normal((n * n, d_v)).astype(np.float32)
    if dtype == "bf16":
        q, C, V = synth.f32_to_bf16(qf), synth.f32_to_bf16(Cf), synth.f32_to_bf16(Vf)
    else:
        q, C, V = qf, Cf, Vf
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=d_v, k=k, dtype=dtype)
    out, idx, w = run_forward(c, q.ravel(), C.ravel(), V.ravel(), form=form)
    ref = oracle.lookup(q.ravel(), C.ravel(), B, H, d_q, n, k)
    assert np.array_equal(idx, ref["idx"])
    assert (np.abs(w - ref["w"]) <= 1e-6 * (1 + ref["w"])).all()


@pytest.mark.parametrize("form", [1, 2, 3])
def test_exact_integer_ties_many_chunks(form):
    # exact ties across chunks and at the KL-th score of long rows: integer
    # scores over 520 subkeys (three 256-key chunks) with runs of duplicated
    # subkey rows, k = 32; every row logs far more than its KL entries, so
    # compactions cut through tied scores
    rng = np.random.default_rng(11)
    B, H, d_q, n, d_v, k = 300, 1, 64, 520, 32, 32
    qf = rng.integers(-2, 3, (B, H, d_q)).astype(np.float32)
    Cf = rng.integers(-1, 2, (H, 2, n, d_q // 2)).astype(np.float32)
    Cf[:, 0, 300:400] = Cf[:, 0, 0:100]
    Cf[:, 1, 256:512] = Cf[:, 1, 0:256]
    Vf = rng.standard_normal((n * n, d_v)).astype(np.float32)
    q, C, V = synth.f32_to_bf16(qf), synth.f32_to_bf16(Cf), synth.f32_to_bf16(Vf)
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=d_v, k=k, dtype="bf16")
    for z in (None, -1e30):
        _, idx, w = run_forward(c, q.ravel(), C.ravel(), V.ravel(), form=form, hint_z=z)
        ref = oracle.lookup(q.ravel(), C.ravel(), B, H, d_q, n, k)
        assert np.array_equal(idx, ref["idx"]), z
        assert (np.abs(w - ref["w"]) <= 1e-6 * (1 + ref["w"])).all(), z


def test_merge_ties_inside_and_at_the_cut_bit_exact():
    # Equal pair sums inside the best k, and at the k-th sum with one or two
    # and with many more pairs reaching it.  Each query's half scores are an
    # integer column pair of the subkeys, 16 c[2m] + c[2m+1] (exact in bf16
    # and fp32), and the 1024 queries take every pair of columns of the two
    # halves.  The order of equal sums (lower flat index first) and the pairs
    # kept at the cut must match the oracle bit for bit.
    rng = np.random.default_rng(21)
    B, H, n, hd, d_v, k = 1024, 1, 64, 64, 32, 32
    d_q = 2 * hd
    Cf = np.zeros((H, 2, n, hd), np.float32)
    for hf in range(2):
        for m in range(hd // 2):
            spread = (2, 8, 40, 127)[m % 4]  # narrow spreads tie often
            Cf[0, hf, :, 2 * m] = rng.integers(-spread, spread + 1, n)
            Cf[0, hf, :, 2 * m + 1] = rng.integers(-127, 128, n)
    qf = np.zeros((B, H, d_q), np.float32)
    for b in range(B):
        m1, m2 = divmod(b, hd // 2)
        qf[b, 0, 2 * m1], qf[b, 0, 2 * m1 + 1] = 16, 1
        qf[b, 0, hd + 2 * m2], qf[b, 0, hd + 2 * m2 + 1] = 16, 1
    # coverage: how many pairs reach the k-th sum of the pruned candidate grid
    kinds = {"distinct": 0, "equal inside": 0, "cut by one or two": 0, "cut by more": 0}
    cand = [(i, j) for i in range(k) for j in range(k) if (i + 1) * (j + 1) <= k]
    ci, cj = np.array(cand).T
    for b in range(B):
        m1, m2 = divmod(b, hd // 2)
        s1 = 16 * Cf[0, 0, :, 2 * m1] + Cf[0, 0, :, 2 * m1 + 1]
        s2 = 16 * Cf[0, 1, :, 2 * m2] + Cf[0, 1, :, 2 * m2 + 1]
        X = s1[np.lexsort((np.arange(n), -s1))[:k]]
        Y = s2[np.lexsort((np.arange(n), -s2))[:k]]
        S = X[ci] + Y[cj]
        top = -np.sort(-S)[:k]
        reach = int((S >= top[-1]).sum())
        kinds["cut by more" if reach > k + 2 else "cut by one or two" if reach > k else
              "equal inside" if (top[1:] == top[:-1]).any() else "distinct"] += 1
    assert min(kinds.values()) >= 10, kinds
    Vf = rng.standard_normal((n * n, d_v)).astype(np.float32)
    q, C, V = synth.f32_to_bf16(qf), synth.f32_to_bf16(Cf), synth.f32_to_bf16(Vf)
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=d_v, k=k, dtype="bf16")
    _, idx, w = run_forward(c, q.ravel(), C.ravel(), V.ravel())
    ref = oracle.lookup(q.ravel(), C.ravel(), B, H, d_q, n, k)
    assert np.array_equal(idx, ref["idx"])
    assert (np.abs(w - ref["w"]) <= 1e-6 * (1 + ref["w"])).all()


def test_gather_alone_fed_oracle_selection():
    # Step a6 in isolation: oracle indices and weights in, fp64 read out.
    for name in ("tiny", "mid"):
        c, q, C, V = cfg_inputs(name)
        B, H, d_q, n, d_v, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "d_v", "k"))
        ref = oracle.lookup(q, C, B, H, d_q, n, k)
        w32 = ref["w"].astype(np.float32)
        expect = oracle.gather(V, n * n, d_v, ref["idx"], w32.astype(np.float64))
        h, _ = make_handle(c)
        try:
            out = torch.empty(B, d_v, device="cuda")
            pk.check(pk.pkm_gather(h, to_device(V, c["dtype"]), B, H, n, k,
                                   torch.from_numpy(ref["idx"]).cuda(),
                                   torch.from_numpy(w32).cuda(), out), "gather")
            assert pk.pkm_get_status(h) == pk.PKM_OK
            got = out.cpu().numpy().astype(np.float64)
        finally:
            pk.pkm_destroy(h)
        assert (np.abs(got - expect) <= 1e-5 * (1 + np.abs(expect))).all(), name


def test_gather_closed_form_ones_and_bad_index():
    B, H, k, n, d_v = 50, 3, 4, 16, 512
    c = dict(B=B, H=H, d_q=32, n_keys=n, d_v=d_v, k=k, dtype="bf16")
    h, _ = make_handle(c)
    try:
        V = torch.ones(n * n, d_v, dtype=torch.bfloat16, device="cuda")
        idx = torch.randint(0, n * n, (B, H, k), device="cuda")
        w = torch.full((B, H, k), 1.0 / k, device="cuda")
        out = torch.empty(B, d_v, device="cuda")
        pk.check(pk.pkm_gather(h, V, B, H, n, k, idx, w, out), "gather")
        assert pk.pkm_get_status(h) == pk.PKM_OK
        torch.testing.assert_close(out, torch.full_like(out, float(H)), rtol=1e-6, atol=1e-6)
        idx[3, 1, 2] = n * n          # out of range: skipped and reported
        idx[7, 0, 0] = -1
        pk.check(pk.pkm_gather(h, V, B, H, n, k, idx, w, out), "gather")
        assert pk.pkm_get_status(h) == pk.PKM_ERR_BAD_INDEX
        assert pk.pkm_get_status(h) == pk.PKM_OK  # reading resets the word
        assert abs(out[3, 0].item() - (H - 1.0 / k)) < 1e-6
    finally:
        pk.pkm_destroy(h)


def test_empty_batch_and_argument_errors():
    c = dict(B=8, H=1, d_q=64, n_keys=32, d_v=64, k=4, dtype="bf16")
    h, cfg = make_handle(c)
    try:
        t = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
        o = torch.zeros(64, dtype=torch.float32, device="cuda")
        assert pk.pkm_forward(h, t, t, t, 0, 1, 32, 4, o) == pk.PKM_OK       # B = 0: no-op
        assert pk.pkm_forward(h, t, t, t, 9, 1, 32, 4, o) == pk.PKM_ERR_RANGE  # B > max_B
        assert pk.pkm_forward(h, t, t, t, 1, 1, 32, 33, o) == pk.PKM_ERR_RANGE
        assert pk.pkm_forward(h, None, t, t, 1, 1, 32, 4, o) == pk.PKM_ERR_INVALID
        assert pk.pkm_forward(h, t.data_ptr() + 2, t, t, 1, 1, 32, 4, o) == pk.PKM_ERR_ALIGN
        assert pk.pkm_forward_host(h, np.zeros(64, np.uint16), t, t, 1, 1, 32, 4,
                                   np.zeros(64, np.float32)) == pk.PKM_ERR_NO_STAGING
        assert pk.pkm_get_status(h) == pk.PKM_OK
    finally:
        pk.pkm_destroy(h)


def test_forward_host_matches_device_forward():
    c, q, C, V = cfg_inputs("mid")
    B = 1000
    c = dict(c, B=B)
    q = q[: B * c["H"] * c["d_q"]]
    out_d, idx_d, w_d = run_forward(c, q, C, V)
    h, _ = make_handle(c, staging=True)
    try:
        qh = torch.from_numpy(q.view(np.int16)).pin_memory()
        dC, dV = to_device(C, "bf16"), to_device(V, "bf16")
        for chunks in (None, 1, 2, 3, 4, 16):  # batch slices pipelined against the copies
            if chunks is not None:
                pk.check(pk.pkm_set_option(h, pk.PKM_OPT_HOST_CHUNKS, chunks), "set_option")
            oh = torch.empty(B, c["d_v"]).pin_memory()
            ih = torch.empty(B, c["H"], c["k"], dtype=torch.int64).pin_memory()
            wh = torch.empty(B, c["H"], c["k"]).pin_memory()
            pk.check(pk.pkm_forward_host(h, qh, dC, dV, B, c["H"], c["n_keys"], c["k"], oh, ih,
                                         wh), "forward_host")
            assert np.array_equal(ih.numpy(), idx_d), chunks
            assert np.array_equal(wh.numpy(), w_d), chunks
            assert np.array_equal(oh.numpy(), out_d), chunks
        # several calls in flight (the handle's three staging slots in turn,
        # and the fourth and fifth calls waiting for the first and second
        # calls' copies back), alternating two query batches and their own
        # output buffers
        q2 = synth.queries(c, rows=B, row_offset=B)
        out_d2, idx_d2, w_d2 = run_forward(c, q2, C, V)
        qh2 = torch.from_numpy(q2.view(np.int16)).pin_memory()
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_HOST_CHUNKS, 3), "set_option")
        h_default, _ = make_handle(c, staging=True)  # async default: one slice
        calls = []
        for i in range(8):
            hh = h if i < 5 else h_default
            oh = torch.empty(B, c["d_v"]).pin_memory()
            ih = torch.empty(B, c["H"], c["k"], dtype=torch.int64).pin_memory()
            ev = torch.cuda.Event()
            pk.check(pk.pkm_forward_host_async(hh, qh if i % 2 == 0 else qh2, dC, dV, B, c["H"],
                                               c["n_keys"], c["k"], oh, ev, ih), "async")
            calls.append((i, oh, ih, ev))
        for i, oh, ih, ev in calls:
            ev.synchronize()
            want_o, want_i = (out_d, idx_d) if i % 2 == 0 else (out_d2, idx_d2)
            assert np.array_equal(ih.numpy(), want_i), i
            assert np.array_equal(oh.numpy(), want_o), i
        pk.pkm_destroy(h_default)
        assert pk.pkm_forward_host_async(h, qh, dC, dV, B, c["H"], c["n_keys"], c["k"], oh,
                                         0) == pk.PKM_ERR_INVALID
        assert pk.pkm_set_option(h, pk.PKM_OPT_HOST_CHUNKS, 0) == pk.PKM_ERR_OPTION
        assert pk.pkm_set_option(h, pk.PKM_OPT_HOST_CHUNKS, 17) == pk.PKM_ERR_OPTION
    finally:
        pk.pkm_destroy(h)


def test_forward_with_scratch_selection_matches():
    # idx/w == NULL: the handle's scratch holds the selection.
    c, q, C, V = cfg_inputs("tiny")
    out_a, _, _ = run_forward(c, q, C, V)
    h, _ = make_handle(c)
    try:
        out = torch.empty(c["B"], c["d_v"], device="cuda")
        pk.check(pk.pkm_forward(h, to_device(q, "f32"), to_device(C, "f32"), to_device(V, "f32"),
                                c["B"], c["H"], c["n_keys"], c["k"], out), "forward")
        assert np.array_equal(out.cpu().numpy(), out_a)
    finally:
        pk.pkm_destroy(h)


def test_multicast_check_on_device_and_host_buffers():
    # device memory of this GPU passes; pinned host memory does not (the
    # one-SM pair form and the query network then take their one-CTA forms)
    import ctypes
    L = pk.lib()
    x = torch.zeros(64, device="cuda")
    y = torch.zeros(64).pin_memory()
    both = (ctypes.c_void_p * 2)(x.data_ptr(), x.data_ptr())
    mixed = (ctypes.c_void_p * 2)(x.data_ptr(), y.data_ptr())
    assert L.pkm_multicast_ok(both, 2) == 1
    assert L.pkm_multicast_ok(mixed, 2) == 0
