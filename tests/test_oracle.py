"""Pins for the fp64 oracle, each independent of the oracle's own code.

Product-Key Memory, "Factorising the key space": the factorised search is
exact, so it must equal a brute-force top-k over every full key.  Memory
Retrieval Mechanisms, top-k retrieval: softmax over the winners, weighted sum
of their value rows.  Cases: brute force, hand-worked numbers, closed forms,
exact integer ties, textbook special cases (k = 1 is an argmax, k = n_keys
reaches every key), and the page's printed operation counts.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(rng, B, H, d_q, n, scale=1.0):
    q = rng.standard_normal((B, H, d_q)).astype(np.float32)
    C = (rng.standard_normal((H, 2, n, d_q // 2)) * scale).astype(np.float32)
    return q, C


def brute_python(q, C, k):
    """Pure-Python exact brute force for integer-valued inputs (no rounding)."""
    B, H, d_q = q.shape
    n = C.shape[2]
    hd = d_q // 2
    res = np.empty((B, H, k), np.int64)
    for b in range(B):
        for h in range(H):
            qq = [int(x) for x in q[b, h]]
            keys = []
            for a in range(n):
                for c in range(n):
                    key = [int(x) for x in C[h, 0, a]] + [int(x) for x in C[h, 1, c]]
                    s = sum(x * y for x, y in zip(qq, key))
                    keys.append((-s, a * n + c))
            keys.sort()
            res[b, h] = [f for _, f in keys[:k]]
    return res


def test_hand_worked_example():
    # d_q = 2 (one element per half), n_keys = 3, k = 2.
    # s1 = q1 * C1 = 2 * [1, 3, 2] = [2, 6, 4];  s2 = q2 * C2 = 1 * [0, -1, 5].
    # Per-half top-2: half 1 -> a = 1 (6), a = 2 (4); half 2 -> b = 2 (5), b = 0 (0).
    # Candidates: (1,2) 11 flat 5; (1,0) 6 flat 3; (2,2) 9 flat 8; (2,0) 4 flat 6.
    # Top-2: flat 5 (11), flat 8 (9).  Softmax: 1/(1+e^-2), e^-2/(1+e^-2).
    q = np.array([[[2.0, 1.0]]], np.float32)
    C = np.array([[[[1.0], [3.0], [2.0]], [[0.0], [-1.0], [5.0]]]], np.float32)
    r = oracle.lookup(q, C, 1, 1, 2, 3, 2)
    assert r["idx"].tolist() == [[[5, 8]]]
    assert r["score"].tolist() == [[[11.0, 9.0]]]
    w0 = 1.0 / (1.0 + math.exp(-2.0))
    assert r["w"][0, 0, 0] == pytest.approx(w0, abs=1e-15)
    assert r["w"][0, 0, 1] == pytest.approx(1.0 - w0, abs=1e-15)
    # value row r = [r, 1]: out = w0 * [5, 1] + (1 - w0) * [8, 1]
    V = np.array([[float(r_), 1.0] for r_ in range(9)], np.float32)
    out = oracle.gather(V, 9, 2, r["idx"], r["w"])
    assert out[0, 0] == pytest.approx(5 * w0 + 8 * (1 - w0), abs=1e-14)
    assert out[0, 1] == pytest.approx(1.0, abs=1e-15)


def test_factorised_equals_brute_force_tiny():
    cfg = synth.CONFIGS["tiny"]
    q, C = synth.queries(cfg), synth.subkeys(cfg)
    args = (cfg["B"], cfg["H"], cfg["d_q"], cfg["n_keys"])
    for k in (1, 2, 8, 17, 32):
        r = oracle.lookup(q, C, *args, k)
        bi, bs = oracle.brute_topk(q, C, *args, k)
        assert np.array_equal(r["idx"], bi), k
        np.testing.assert_allclose(r["score"], bs, rtol=0, atol=1e-12)


def test_factorised_equals_brute_force_multihead_random():
    rng = np.random.default_rng(11)
    q, C = rand_problem(rng, 6, 3, 10, 9)
    r = oracle.lookup(q, C, 6, 3, 10, 9, 5)
    bi, _ = oracle.brute_topk(q, C, 6, 3, 10, 9, 5)
    assert np.array_equal(r["idx"], bi)


def test_factorised_equals_brute_force_mid_sampled_bf16():
    cfg = synth.CONFIGS["mid"]
    rows = 3
    q = synth.queries(cfg, rows=rows, row_offset=1000)
    C = synth.subkeys(cfg)
    args = (rows, cfg["H"], cfg["d_q"], cfg["n_keys"], cfg["k"])
    r = oracle.lookup(q, C, *args, want_gaps=True)
    bi, bs = oracle.brute_topk(q, C, *args)
    # identical unless two keys are within fp64 rounding of each other
    same = (r["idx"] == bi).all(axis=-1)
    assert same.all() or (r["gap_in"][~same].min() < 1e-12)
    np.testing.assert_allclose(r["score"], bs, rtol=1e-12, atol=1e-12)


def test_integer_ties_exact():
    # Small integers are exact in fp32 and fp64, so every score is exact and
    # duplicated subkey rows force exact ties; the rule is lower flat index.
    rng = np.random.default_rng(5)
    B, H, d_q, n = 4, 2, 6, 7
    q = rng.integers(-2, 3, (B, H, d_q)).astype(np.float32)
    C = rng.integers(-2, 3, (H, 2, n, d_q // 2)).astype(np.float32)
    C[:, 0, 4] = C[:, 0, 1]  # duplicate rows -> ties in half 1
    C[:, 1, 6] = C[:, 1, 0]  # and in half 2
    for k in (1, 3, 7):
        r = oracle.lookup(q, C, B, H, d_q, n, k)
        assert np.array_equal(r["idx"], brute_python(q, C, k)), k


def test_all_equal_scores_pick_lowest_flat():
    # Zero subkeys: every key scores 0, so the answer is flat 0..k-1, uniform w.
    q = np.ones((2, 1, 8), np.float32)
    C = np.zeros((1, 2, 5, 4), np.float32)
    r = oracle.lookup(q, C, 2, 1, 8, 5, 4, want_gaps=True)
    assert r["idx"].tolist() == [[[0, 1, 2, 3]]] * 2
    np.testing.assert_allclose(r["w"], 0.25, rtol=0, atol=1e-15)
    assert (r["gap_k"] == 0).all()


def test_k1_is_argmax():
    rng = np.random.default_rng(3)
    B, H, d_q, n = 20, 2, 16, 11
    q, C = rand_problem(rng, B, H, d_q, n)
    r = oracle.lookup(q, C, B, H, d_q, n, 1)
    qd, Cd = q.astype(np.float64), C.astype(np.float64)
    s1 = np.einsum("bht,hat->bha", qd[..., : d_q // 2], Cd[:, 0])
    s2 = np.einsum("bht,hat->bha", qd[..., d_q // 2:], Cd[:, 1])
    expect = s1.argmax(-1) * n + s2.argmax(-1)
    assert np.array_equal(r["idx"][..., 0], expect)
    assert (r["w"] == 1.0).all()


def test_k_equals_nkeys_reaches_every_key():
    # k = n_keys: the k^2 candidate set is the whole key space.
    rng = np.random.default_rng(8)
    q, C = rand_problem(rng, 3, 1, 8, 6)
    r = oracle.lookup(q, C, 3, 1, 8, 6, 6)
    qd, Cd = q.astype(np.float64), C.astype(np.float64)
    for b in range(3):
        s1 = Cd[0, 0] @ qd[b, 0, :4]
        s2 = Cd[0, 1] @ qd[b, 0, 4:]
        full = (s1[:, None] + s2[None, :]).ravel()
        order = sorted(range(36), key=lambda f: (-full[f], f))[:6]
        assert r["idx"][b, 0].tolist() == order


def test_softmax_invariants():
    cfg = synth.CONFIGS["tiny"]
    q, C = synth.queries(cfg), synth.subkeys(cfg)
    r = oracle.lookup(q, C, 64, 1, 64, 32, 8)
    np.testing.assert_allclose(r["w"].sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (np.diff(r["w"], axis=-1) <= 0).all()
    assert (np.diff(r["score"], axis=-1) <= 0).all()
    # closed form: w_j = exp(s_j) / sum exp(s_l)
    e = np.exp(r["score"] - r["score"][..., :1])
    np.testing.assert_allclose(r["w"], e / e.sum(-1, keepdims=True), rtol=1e-13)


def test_gather_closed_forms():
    rng = np.random.default_rng(1)
    B, H, k, N, d = 5, 3, 4, 64, 64
    idx = rng.integers(0, N, (B, H, k)).astype(np.int64)
    w = rng.random((B, H, k))
    w /= w.sum(-1, keepdims=True)
    ones = np.ones((N, d), np.float32)
    np.testing.assert_allclose(oracle.gather(ones, N, d, idx, w), float(H), atol=1e-14)
    ramp = np.repeat(np.arange(N, dtype=np.float32)[:, None], d, 1)
    expect = (w * idx).sum((1, 2))
    np.testing.assert_allclose(oracle.gather(ramp, N, d, idx, w), expect[:, None] * np.ones(d),
                               rtol=1e-14)
    onehot = np.zeros((N, d), np.float32)
    onehot[np.arange(N), np.arange(N) % d] = 1.0
    scat = np.zeros((B, d))
    for b in range(B):
        for h in range(H):
            for j in range(k):
                scat[b, idx[b, h, j] % d] += w[b, h, j]
    np.testing.assert_allclose(oracle.gather(onehot, N, d, idx, w), scat, atol=1e-15)
    # bf16 bits widen exactly: 1.0 = 0x3F80
    onesb = np.full((N, d), 0x3F80, np.uint16)
    np.testing.assert_allclose(oracle.gather(onesb, N, d, idx, w), float(H), atol=1e-14)


def test_gather_rejects_out_of_range_index():
    V = np.ones((4, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.gather(V, 4, 2, np.array([[[4]]], np.int64), np.array([[[1.0]]]))


def test_forward_matches_torch_sketch_float64():
    # The page's module forward, run op by op in float64 torch on continuous
    # inputs (no ties): chunk, per-half matmul + topk, k^2 sums, flat index
    # i1 * n + i2, topk, softmax, weighted sum of value rows; heads summed.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    B, H, d_q, n, d_v, k = 7, 2, 12, 9, 5, 4
    q, C = rand_problem(rng, B, H, d_q, n)
    V = rng.standard_normal((n * n, d_v)).astype(np.float32)
    idx, w, out = oracle.forward(q, C, V, B, H, d_q, n, d_v, k)
    tq, tC, tV = (torch.from_numpy(x).double() for x in (q, C, V))
    tout = torch.zeros(B, d_v, dtype=torch.float64)
    for h in range(H):
        q1, q2 = tq[:, h].chunk(2, dim=-1)
        s1, i1 = (q1 @ tC[h, 0].T).topk(k)
        s2, i2 = (q2 @ tC[h, 1].T).topk(k)
        scores = (s1[:, :, None] + s2[:, None, :]).flatten(1)
        flat = (i1[:, :, None] * n + i2[:, None, :]).flatten(1)
        top, pos = scores.topk(k)
        sel = flat.gather(1, pos)
        wt = top.softmax(-1)
        assert np.array_equal(sel.numpy(), idx[:, h])
        np.testing.assert_allclose(wt.numpy(), w[:, h], rtol=1e-12)
        tout += (wt[:, :, None] * tV[sel]).sum(1)
    np.testing.assert_allclose(out, tout.numpy(), rtol=1e-12, atol=1e-14)


def test_page_operation_counts():
    g = json.load(open(os.path.join(GOLDEN, "page_op_counts.json")))
    n, k = g["n_keys"], g["k"]
    rng = np.random.default_rng(2)
    q, C = rand_problem(rng, 1, 1, 4, n)
    r = oracle.lookup(q, C, 1, 1, 4, n, k)
    assert r["counters"][0] == g["subkey_comparisons"]  # 2 sqrt(N) per query and head
    assert r["counters"][1] == g["merge_candidates"] == k * k
    # "instead of a million": the flat search scores every one of n^2 keys
    assert abs(n * n - g["flat_comparisons_approx"]) / g["flat_comparisons_approx"] < 0.05
    assert abs(g["value_params_N"] * g["value_params_d"] - g["value_params_approx"]) \
        / g["value_params_approx"] < 0.05
    # top-k retrieval: k / n_slots; 0.05% at k = 5 implies 10^4 slots
    slots = 5 / (g["topk_fraction_k5_percent"] / 100)
    assert round(slots / 5) == g["topk_reduction_k5"]
    assert 100 * 100 / slots == g["topk_fraction_k100_percent"]


def test_near_tie_report():
    # Make the k-th and (k+1)-th full keys tie exactly: duplicate a half-2 subkey.
    q = np.array([[[1.0, 0.0, 1.0, 0.0]]], np.float32)
    C = np.zeros((1, 2, 4, 2), np.float32)
    C[0, 0, :, 0] = [4.0, 3.0, 2.0, 1.0]
    C[0, 1, :, 0] = [0.5, 0.25, 0.25, -9.0]
    r = oracle.lookup(q, C, 1, 1, 4, 4, 2, want_gaps=True)
    # best: (0,0)=4.5 flat 0; next (0,1) and (0,2) tie at 4.25 -> flat 1 wins
    assert r["idx"].tolist() == [[[0, 1]]]
    assert r["gap_k"][0, 0] == 0.0
    assert r["gap_in"][0, 0] == pytest.approx(0.25 / 4.5)


def test_rejects_bad_shapes():
    q = np.zeros((1, 1, 4), np.float32)
    C = np.zeros((1, 2, 3, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.lookup(q, C, 1, 1, 4, 3, 4)  # k > n_keys
    with pytest.raises(ValueError):
        oracle.lookup(q, C, 1, 1, 3, 3, 1)  # odd d_q


# ------------------------------------------------------------------ fp8 table
#
# Product-Key Memory, note after the code listing: the value table is "a good
# candidate for keeping in a lower precision".  The fp8 e4m3 format (OCP 8-bit
# floating point: bias 7, 3 mantissa bits, subnormals, S.1111.111 = NaN, no
# infinities) is pinned against torch's float8_e4m3fn and against brute force
# over its finite values; the quantiser and the fp8 read against closed forms.

def _finite_e4m3():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    return codes, np.array([oracle.e4m3_value(c) for c in codes])


def test_e4m3_values_match_torch_for_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mine = np.array([oracle.e4m3_value(c) for c in codes])
    assert (np.isnan(ref) == np.isnan(mine)).all()
    fin = ~np.isnan(ref)
    assert (ref[fin] == mine[fin]).all()
    # a few values from the definition itself
    assert oracle.e4m3_value(0x01) == 2.0 ** -9 and oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0xFE) == -448.0


def test_e4m3_encode_is_nearest_with_ties_to_even():
    torch = pytest.importorskip("torch")
    codes, vals = _finite_e4m3()
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * rng.choice([1e-3, 0.05, 1.0, 40.0, 300.0], 4000))
    x = x.astype(np.float32)
    # exact midpoints between neighbours, both signs
    pos = np.sort(vals[vals > 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 2.0 ** -10, 447.0])])
    x = x[np.abs(x) < 448]
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    # brute force: nearest finite value, ties to the even code (even mantissa)
    for v, g in zip(x[:1500], got[:1500]):
        d = np.abs(vals - float(v))
        best = d.min()
        cand = [c for c, dd in zip(codes, d) if dd == best]
        same_sign = [c for c in cand if (c >> 7) == (1 if np.signbit(v) else 0)]
        cand = same_sign or cand
        want = [c for c in cand if (c & 1) == 0] if len(cand) > 1 else cand
        assert g == want[0], (v, g, cand)
    # and torch's round-to-nearest-even cast agrees on every in-range value
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got == ref).all()


def test_e4m3_encode_saturates():
    for v in (448.0, 460.0, 464.0, 470.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_quantize_fp8_scales_and_error_bound():
    rng = np.random.default_rng(6)
    N, d_v = 300, 48
    V = (rng.standard_normal((N, d_v)) * rng.choice([1e-30, 1e-4, 1.0, 1e4], (N, 1)))
    V = V.astype(np.float32)
    V[7] = 0.0                      # an all-zero row
    V[8, :] = 0.0
    V[8, 3] = -2.5                  # a single non-zero element
    codes, scales = oracle.quantize_fp8(V, N, d_v)
    amax = np.abs(V).max(axis=1)
    want_scale = np.maximum(amax / np.float32(448.0), np.finfo(np.float32).tiny)
    assert (scales == want_scale.astype(np.float32)).all()
    dq = np.vectorize(oracle.e4m3_value)(codes) * scales[:, None].astype(np.float64)
    # e4m3: relative spacing 2^-3 for normals -> half a step = 2^-4 of the value;
    # below 2^-6 the step is 2^-9 (absolute, in units of the scale)
    bound = np.maximum(np.abs(V) * 2.0 ** -4, 2.0 ** -10 * scales[:, None])
    assert (np.abs(dq - V) <= bound * (1 + 1e-12)).all()
    assert (codes[7] == 0).all() and (dq[7] == 0).all()
    # the row's only value maps to -448; the scale 2.5 / 448 is rounded to fp32
    assert codes[8, 3] == 0xFE and abs(dq[8, 3] + 2.5) <= 2.5 * 2.0 ** -24
    # every non-zero row's largest magnitude lands on +-448
    for r in range(N):
        if amax[r] > 0:
            c = codes[r, np.argmax(np.abs(V[r]))]
            assert c & 0x7F == 0x7E


def test_quantize_fp8_bf16_input_matches_fp32_input():
    rng = np.random.default_rng(7)
    V = synth.normal(3, 3, 64 * 32, 0.5, dtype="bf16").reshape(64, 32)
    V32 = (V.astype(np.uint32) << 16).view(np.float32)
    a = oracle.quantize_fp8(V, 64, 32)
    b = oracle.quantize_fp8(V32, 64, 32)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all()


def test_gather_fp8_closed_forms():
    rng = np.random.default_rng(8)
    B, H, k, d_v, N = 5, 3, 4, 32, 96
    idx = rng.integers(0, N, (B, H, k)).astype(np.int64)
    w = rng.random((B, H, k))
    w /= w.sum(-1, keepdims=True)
    # every code 1.0 with scale 1 -> out = H everywhere
    out = oracle.gather_fp8(np.full((N, d_v), 0x38, np.uint8), np.ones(N, np.float32), N, d_v,
                            idx, w)
    np.testing.assert_allclose(out, H, rtol=0, atol=1e-12)
    # one-hot rows: row r holds 1.0 at column r mod d_v, scaled by s_r
    codes = np.zeros((N, d_v), np.uint8)
    codes[np.arange(N), np.arange(N) % d_v] = 0x38
    s = (1.0 + np.arange(N) / 8).astype(np.float32)
    out = oracle.gather_fp8(codes, s, N, d_v, idx, w)
    want = np.zeros((B, d_v))
    for b in range(B):
        for h in range(H):
            for j in range(k):
                want[b, idx[b, h, j] % d_v] += w[b, h, j] * float(s[idx[b, h, j]])
    np.testing.assert_allclose(out, want, rtol=1e-14, atol=0)
    with pytest.raises(ValueError):
        bad = idx.copy()
        bad[0, 0, 0] = N
        oracle.gather_fp8(codes, s, N, d_v, bad, w)


# ----------------------------------------------------------- query network
#
# Product-Key Memory, code listing: q = BatchNorm1d(Linear(dim, F, bias=False)(x)),
# the BatchNorm in its inference form (running statistics).

def test_query_net_matches_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    B, dim, F, eps = 37, 48, 96, 1e-5
    x = rng.standard_normal((B, dim)).astype(np.float32)
    W = (rng.standard_normal((F, dim)) / np.sqrt(dim)).astype(np.float32)
    gamma = (1 + 0.2 * rng.standard_normal(F)).astype(np.float32)
    beta = (0.3 * rng.standard_normal(F)).astype(np.float32)
    mean = (0.1 * rng.standard_normal(F)).astype(np.float32)
    var = (0.5 + rng.random(F)).astype(np.float32)
    q = oracle.query_net(x, W, B, dim, F, gamma, beta, mean, var, eps)
    lin = torch.nn.Linear(dim, F, bias=False).double()
    bn = torch.nn.BatchNorm1d(F, eps=eps).double().eval()
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(W.astype(np.float64)))
        bn.weight.copy_(torch.from_numpy(gamma.astype(np.float64)))
        bn.bias.copy_(torch.from_numpy(beta.astype(np.float64)))
        bn.running_mean.copy_(torch.from_numpy(mean.astype(np.float64)))
        bn.running_var.copy_(torch.from_numpy(var.astype(np.float64)))
        ref = bn(lin(torch.from_numpy(x.astype(np.float64)))).numpy()
    np.testing.assert_allclose(q, ref, rtol=1e-12, atol=1e-12)


def test_query_net_closed_forms():
    rng = np.random.default_rng(32)
    B, dim = 9, 32
    x = rng.standard_normal((B, dim)).astype(np.float32)
    eye = np.eye(dim, dtype=np.float32)
    one, zero = np.ones(dim, np.float32), np.zeros(dim, np.float32)
    # identity weight, neutral normalisation (var + eps = 1): q = x
    q = oracle.query_net(x, eye, B, dim, dim, one, zero, zero, np.full(dim, 0.75, np.float32), 0.25)
    assert (q == x.astype(np.float64)).all()
    # identity weight: q = (x - mean) / sqrt(var + eps) * gamma + beta, column by column
    g, bt, m, v = (rng.random(dim).astype(np.float32) + 0.5 for _ in range(4))
    q = oracle.query_net(x, eye, B, dim, dim, g, bt, m, v, 1e-3)
    want = (x.astype(np.float64) - m) / np.sqrt(v.astype(np.float64) + 1e-3) * g + bt
    np.testing.assert_allclose(q, want, rtol=1e-14)
    # a bf16 input gives the same result as its exact fp32 widening
    xb = synth.normal(5, 6, B * dim, 1.0, dtype="bf16").reshape(B, dim)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    a = oracle.query_net(xb, eye, B, dim, dim, g, bt, m, v, 1e-3)
    b = oracle.query_net(xf, eye, B, dim, dim, g, bt, m, v, 1e-3)
    assert (a == b).all()


# The BatchNorm in training mode ("Product-Key Memory", "Keeping the memory in
# use": the batch's own statistics normalise the queries).

def test_query_net_batch_matches_torch_float64_train_mode():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    B, dim, F, eps = 53, 40, 72, 1e-5
    x = rng.standard_normal((B, dim)).astype(np.float32)
    # features with a large common offset: the variance must not come from
    # the difference of two large sums
    x[:, 0] += 300.0
    W = (rng.standard_normal((F, dim)) / np.sqrt(dim)).astype(np.float32)
    gamma = (1 + 0.2 * rng.standard_normal(F)).astype(np.float32)
    beta = (0.3 * rng.standard_normal(F)).astype(np.float32)
    q, mean, var = oracle.query_net_batch(x, W, B, dim, F, gamma, beta, eps)
    lin = torch.nn.Linear(dim, F, bias=False).double()
    # momentum 1: the running statistics become the batch's (variance unbiased)
    bn = torch.nn.BatchNorm1d(F, eps=eps, momentum=1.0).double().train()
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(W.astype(np.float64)))
        bn.weight.copy_(torch.from_numpy(gamma.astype(np.float64)))
        bn.bias.copy_(torch.from_numpy(beta.astype(np.float64)))
        ref = bn(lin(torch.from_numpy(x.astype(np.float64)))).numpy()
    np.testing.assert_allclose(q, ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(mean, bn.running_mean.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(var, bn.running_var.numpy() * (B - 1) / B, rtol=1e-10)


def test_query_net_batch_invariants_and_special_cases():
    rng = np.random.default_rng(42)
    B, dim, F, eps = 31, 24, 40, 1e-3
    x = rng.standard_normal((B, dim)).astype(np.float32)
    W = rng.standard_normal((F, dim)).astype(np.float32)
    W[5] = 0.0  # a constant (zero) feature
    gamma = (rng.random(F) + 0.5).astype(np.float32)
    beta = rng.standard_normal(F).astype(np.float32)
    q, mean, var = oracle.query_net_batch(x, W, B, dim, F, gamma, beta, eps)
    # every feature leaves with mean beta and biased variance
    # gamma^2 var / (var + eps)
    np.testing.assert_allclose(q.mean(0), beta.astype(np.float64), atol=1e-12)
    want_var = gamma.astype(np.float64) ** 2 * var / (var + eps)
    np.testing.assert_allclose(((q - q.mean(0)) ** 2).mean(0), want_var, rtol=1e-10, atol=1e-14)
    # the constant feature: mean 0, variance 0, q = beta
    assert mean[5] == 0.0 and var[5] == 0.0
    assert (q[:, 5] == np.float64(beta[5])).all()
    # B = 1: variance 0, every feature equals beta
    q1, _, v1 = oracle.query_net_batch(x[:1], W, 1, dim, F, gamma, beta, eps)
    assert (v1 == 0).all() and (q1[0] == beta.astype(np.float64)).all()
    # two rows: mean and variance in closed form
    z = x[:2].astype(np.float64) @ W.astype(np.float64).T
    _, m2, v2 = oracle.query_net_batch(x[:2], W, 2, dim, F, gamma, beta, eps)
    np.testing.assert_allclose(m2, (z[0] + z[1]) / 2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(v2, ((z[0] - z[1]) / 2) ** 2, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ backward
#
# The forward pass is differentiable for a fixed selection (the code listing's
# autograd runs through the selected scores, the softmax and the EmbeddingBag
# read).  The oracle's gradients are pinned by central finite differences of
# L = sum(dout * out) computed with the oracle's own forward on perturbed
# inputs, in fp32-exact problems whose selection does not change.

def _loss(q, C, V, B, H, d_q, n, d_v, k, dout):
    _, _, out = oracle.forward(q, C, V, B, H, d_q, n, d_v, k)
    return float((out * dout).sum())


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(41)
    B, H, d_q, n, d_v, k = 3, 2, 8, 6, 5, 4
    q = rng.standard_normal((B, H, d_q)).astype(np.float32)
    C = rng.standard_normal((H, 2, n, d_q // 2)).astype(np.float32)
    V = rng.standard_normal((n * n, d_v)).astype(np.float32)
    dout = rng.standard_normal((B, d_v))
    ref = oracle.lookup(q, C, B, H, d_q, n, k, want_gaps=True)
    assert ref["gap_k"].min() > 1e-3  # the selection is stable under small steps
    g = oracle.backward(q, C, V, B, H, d_q, n, d_v, k, ref["idx"], ref["w"], dout)
    eps = 1e-3

    def numeric(arr, pos, fn):
        a = arr.copy(); a[pos] += eps
        b = arr.copy(); b[pos] -= eps
        return (fn(a) - fn(b)) / (2 * eps)

    for pos in [(0, 0, 1), (1, 1, 7), (2, 0, 4)]:
        num = numeric(q, pos, lambda a: _loss(a, C, V, B, H, d_q, n, d_v, k, dout))
        assert abs(num - g["dq"][pos]) <= 1e-4 * (1 + abs(num)), (pos, num, g["dq"][pos])
    used = np.unique(ref["idx"])
    for r in used[:3]:
        pos = (int(r), 2)
        num = numeric(V, pos, lambda a: _loss(q, C, a, B, H, d_q, n, d_v, k, dout))
        assert abs(num - g["dvalues"][pos]) <= 1e-4 * (1 + abs(num))
    a1 = int(ref["idx"][0, 0, 0] // n)
    for pos in [(0, 0, a1, 1), (0, 0, a1, 3)]:
        num = numeric(C, pos, lambda a: _loss(q, a, V, B, H, d_q, n, d_v, k, dout))
        assert abs(num - g["dsubkeys"][pos]) <= 1e-4 * (1 + abs(num)), (pos, num)
    # unselected rows and subkeys get nothing
    untouched = np.setdiff1d(np.arange(n * n), used)
    assert (g["dvalues"][untouched] == 0).all()


def test_backward_closed_forms():
    # one selected row (k = 1): w = 1, so ds = 0 and only the read carries
    # gradient: dV[idx] = dout, dq = 0, dsubkeys = 0, dw = dout . V[idx]
    rng = np.random.default_rng(42)
    B, H, d_q, n, d_v = 4, 1, 6, 5, 3
    q = rng.standard_normal((B, H, d_q)).astype(np.float32)
    C = rng.standard_normal((H, 2, n, d_q // 2)).astype(np.float32)
    V = rng.standard_normal((n * n, d_v)).astype(np.float32)
    dout = rng.standard_normal((B, d_v))
    ref = oracle.lookup(q, C, B, H, d_q, n, 1)
    g = oracle.backward(q, C, V, B, H, d_q, n, d_v, 1, ref["idx"], ref["w"], dout)
    want = np.zeros((n * n, d_v))
    for b in range(B):
        want[ref["idx"][b, 0, 0]] += dout[b]
    np.testing.assert_allclose(g["dvalues"], want, rtol=1e-15)
    assert (g["dq"] == 0).all() and (g["dsubkeys"] == 0).all()
    np.testing.assert_allclose(g["dw"][:, 0, 0],
                               (dout * V[ref["idx"][:, 0, 0]].astype(np.float64)).sum(-1))
    # the row-subset form of dvalues returns the same rows (in the order asked)
    rows = [int(ref["idx"][2, 0, 0]), 0, int(ref["idx"][0, 0, 0])]
    rows = list(dict.fromkeys(rows))
    g2 = oracle.backward(q, C, V, B, H, d_q, n, d_v, 1, ref["idx"], ref["w"], dout,
                         dvalue_rows=rows)
    np.testing.assert_array_equal(g2["dvalues"], want[rows])
