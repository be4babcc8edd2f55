"""The flat exact top-k on the GPU (pkm_full_keys + pkm_flat_lookup) against
the oracle's brute force over every full key.

Memory Retrieval Mechanisms, top-k retrieval: score all N keys, keep the k
best, softmax over them.  Product-Key Memory, "Factorising the key space":
a full key is concat(c1_a, c2_b) with flat index a * n_keys + b; the top-k
over all N of them is the top-k the factorised search returns.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_lookup, exact_scores, make_handle, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")


def case(seed, B, H, d_q, n, k):
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=64, k=k, dtype="bf16")
    q = synth.normal(seed, 1, B * H * d_q, 1.0, dtype="bf16")
    C = synth.normal(seed, 2, H * 2 * n * (d_q // 2), 2.0 / d_q, dtype="bf16")
    return c, q, C


def run_flat(c, q, C, also_factorised=False, keys_back=True):
    """Full keys and flat top-k on the GPU; returns (keys bits or None, idx, w[, f_idx,
    f_w])."""
    B, H, d_q, n, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "k"))
    h, _ = make_handle(dict(c, B=max(B, 1)))
    try:
        dq, dC = to_device(q, "bf16"), to_device(C, "bf16")
        keys = torch.empty(H, n * n, d_q, dtype=torch.bfloat16, device="cuda")
        pk.check(pk.pkm_full_keys(h, dC, H, n, keys), "full_keys")
        idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
        w = torch.empty(B, H, k, device="cuda")
        pk.check(pk.pkm_flat_lookup(h, dq, keys, B, H, n, k, idx, w), "flat_lookup")
        res = [keys.view(torch.int16).cpu().numpy().view(np.uint16) if keys_back else None,
               idx.cpu().numpy(), w.cpu().numpy()]
        if also_factorised:
            fi = torch.empty_like(idx)
            fw = torch.empty_like(w)
            pk.check(pk.pkm_lookup(h, dq, dC, B, H, n, k, fi, fw), "lookup")
            res += [fi.cpu().numpy(), fw.cpu().numpy()]
        assert pk.pkm_get_status(h) == pk.PKM_OK
        return res
    finally:
        pk.pkm_destroy(h)


def brute_ref(c, q, C, rows=None):
    """Oracle brute force (idx, score) with the factorised oracle's softmax
    weights (the two oracles select the same keys: pinned in the oracle tests)."""
    B, H, d_q, n, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "k"))
    if rows is not None:
        q = q.reshape(B, H * d_q)[rows].ravel()
        B = len(rows)
    bi, bs = oracle.brute_topk(q, C, B, H, d_q, n, k)
    ref = oracle.lookup(q, C, B, H, d_q, n, k)
    assert np.array_equal(bi, ref["idx"])
    return dict(idx=bi, score=bs, w=ref["w"]), q, B


def test_full_keys_are_the_concatenated_subkeys():
    c, q, C = case(5, 1, 3, 96, 24, 4)
    keys, _, _ = run_flat(c, q, C)
    H, n, hd = 3, 24, 48
    Cb = C.reshape(H, 2, n, hd)
    expect = np.concatenate([np.repeat(Cb[:, 0], n, axis=1), np.tile(Cb[:, 1], (1, n, 1))], -1)
    assert np.array_equal(keys.reshape(H, n * n, 2 * hd), expect)


@pytest.mark.parametrize("shape", [
    # B, H, d_q, n, k
    (64, 1, 64, 32, 8),        # the tiny problem's shapes in bf16: N = 1024 (four chunks)
    (300, 2, 128, 24, 5),      # ragged: 300 rows (one and a bit pair tiles), N = 576
    (257, 3, 96, 40, 32),      # d_q = 96 (a partial k-slab), N = 1600, k = 32
    (40, 1, 32, 20, 1),        # k = 1: the argmax
    (33, 2, 64, 12, 12),       # k = n_keys (the largest k a handle takes), N = 144 < one chunk
    (70, 8, 128, 48, 32),      # eight heads (the skewed workload's H), N = 2304
])
def test_flat_matches_brute_force(shape):
    c, q, C = case(sum(shape), *shape)
    _, idx, w = run_flat(c, q, C)
    ref, _, _ = brute_ref(c, q, C)
    B, H, d_q, n, k = shape
    rep = compare_lookup(idx, w, ref, q, C, "bf16", H, d_q, n)
    assert rep["failures"] == 0, rep
    assert rep["near_ties"] <= 0.01 * B * H, rep
    assert rep["w_ok"], rep
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-5)


def test_flat_exact_integer_ties_bit_exact():
    # integer scores with many exact ties, also across chunks: the lower flat
    # index wins, as in the brute force
    rng = np.random.default_rng(3)
    B, H, d_q, n, k = 200, 2, 64, 40, 32
    qf = rng.integers(-2, 3, (B, H, d_q)).astype(np.float32)
    Cf = rng.integers(-1, 2, (H, 2, n, d_q // 2)).astype(np.float32)
    Cf[:, 1, 30:40] = Cf[:, 1, 0:10]
    q, C = synth.f32_to_bf16(qf).ravel(), synth.f32_to_bf16(Cf).ravel()
    c = dict(B=B, H=H, d_q=d_q, n_keys=n, d_v=64, k=k, dtype="bf16")
    _, idx, w = run_flat(c, q, C)
    ref, _, _ = brute_ref(c, q, C)
    assert np.array_equal(idx, ref["idx"])
    assert (np.abs(w - ref["w"]) <= 1e-6 * (1 + ref["w"])).all()


def test_flat_mid_sampled_against_brute_force_and_factorised():
    # the mid workload in full on the GPU (N = 65536 full keys per head);
    # sampled queries against the oracle's brute force, and every query
    # against the factorised GPU search (same keys outside near-ties)
    c = synth.CONFIGS["mid"]
    q, C = synth.queries(c), synth.subkeys(c)
    B, H, d_q, n, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "k"))
    _, idx, w, fidx, fw = run_flat(dict(c), q, C, also_factorised=True, keys_back=False)
    rows = np.random.default_rng(7).choice(B, 12, replace=False)
    ref, qs, Bs = brute_ref(c, q, C, rows)
    rep = compare_lookup(idx[rows], w[rows], ref, qs, C, "bf16", H, d_q, n)
    assert rep["failures"] == 0 and rep["w_ok"], rep
    fsc = exact_scores(q, C, "bf16", H, d_q, n, fidx)
    rep = compare_lookup(idx, w, dict(idx=fidx, w=fw.astype(np.float64), score=fsc), q, C, "bf16",
                         H, d_q, n)
    assert rep["failures"] == 0, rep
    assert rep["near_ties"] <= 0.01 * B * H, rep
    assert rep["w_ok"], rep


def test_flat_argument_errors():
    c, q, C = case(1, 4, 1, 64, 16, 4)
    h, _ = make_handle(c)
    try:
        dq, dC = to_device(q, "bf16"), to_device(C, "bf16")
        keys = torch.empty(1, 256, 64, dtype=torch.bfloat16, device="cuda")
        idx = torch.empty(4, 1, 4, dtype=torch.int64, device="cuda")
        w = torch.empty(4, 1, 4, device="cuda")
        assert pk.pkm_flat_lookup(h, dq, keys, 0, 1, 16, 4, idx, w) == pk.PKM_OK
        assert pk.pkm_flat_lookup(h, dq, keys, 5, 1, 16, 4, idx, w) == pk.PKM_ERR_RANGE
        assert pk.pkm_flat_lookup(h, dq, None, 4, 1, 16, 4, idx, w) == pk.PKM_ERR_INVALID
        assert pk.pkm_full_keys(h, dC, 1, 16, None) == pk.PKM_ERR_INVALID
        assert pk.pkm_full_keys(h, dC, 1, 17, keys) == pk.PKM_ERR_RANGE
        assert pk.pkm_get_status(h) == pk.PKM_OK
    finally:
        pk.pkm_destroy(h)


def test_flat_page_shapes_small_batch():
    # the page workload's tables at a small batch: N = 2^20 full keys per head
    # (an 8 GiB full key table), d_q = 1024, k = 32; every (query, head) against
    # the factorised GPU search, sampled queries against the oracle (whose
    # factorised search is pinned to its brute force)
    c = dict(synth.CONFIGS["page"], B=256)
    q, C = synth.queries(c), synth.subkeys(c)
    B, H, d_q, n, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "k"))
    _, idx, w, fidx, fw = run_flat(c, q, C, also_factorised=True, keys_back=False)
    fsc = exact_scores(q, C, "bf16", H, d_q, n, fidx)
    rep = compare_lookup(idx, w, dict(idx=fidx, w=fw.astype(np.float64), score=fsc), q, C, "bf16",
                         H, d_q, n)
    assert rep["failures"] == 0, rep
    assert rep["near_ties"] <= 0.01 * B * H, rep
    assert rep["w_ok"], rep
    rows = np.random.default_rng(9).choice(B, 16, replace=False)
    qs = q.reshape(B, H * d_q)[rows].ravel()
    ref = oracle.lookup(qs, C, len(rows), H, d_q, n, k)
    rep = compare_lookup(idx[rows], w[rows], ref, qs, C, "bf16", H, d_q, n)
    assert rep["failures"] == 0 and rep["w_ok"], rep
