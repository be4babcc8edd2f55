"""GPU parity of the two forms of the value read (step a6) against the fp64
oracle, through pkm_gather.

Product-Key Memory (EmbeddingBag note): out[b] = sum over the bag's H*k
selected rows of weight * row.  Rows of 512-byte multiples stream through a
shared-memory ring as whole-row bulk copies (one persistent CTA per SM, the
SM count set by PKM_OPT_READ_SMS); other widths take one CTA per query.  Both
accumulate in fp32, so each output is compared with the oracle's fp64 sum
within 1e-5 * (1 + |ref|).  The cases cover bags whose H*k is not a multiple
of the 8-row copy batch, batches smaller than a CTA's team count, one SM
cycling through every bag (its ring slots and staging buffers reused many
times), fp32, bf16 and fp8 tables, 8 KB rows, and out-of-range indices.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")

DT = {"f32": pk.PKM_F32, "bf16": pk.PKM_BF16, "fp8": pk.PKM_FP8_E4M3}


def read_case(seed, B, H, n, d_v, k, vdt):
    """Random selection (indices anywhere in the table, weights in (0, 1])
    and a seeded value table; returns the device table, the selection and the
    oracle's fp64 read."""
    N = n * n
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, N, (B, H, k)).astype(np.int64)
    w = rng.uniform(0.01, 1.0, (B, H, k)).astype(np.float32)
    if vdt == "fp8":
        V = synth.normal(seed, 3, N * d_v, 1.0, dtype="bf16")
        codes, scales = oracle.quantize_fp8(V, N, d_v)
        table = np.concatenate([codes.ravel(), scales.view(np.uint8)])
        dV = torch.from_numpy(table).cuda()
        ref = oracle.gather_fp8(codes, scales, N, d_v, idx, w.astype(np.float64))
    else:
        V = synth.normal(seed, 3, N * d_v, 1.0, dtype=vdt)
        if vdt == "f32":
            dV = torch.from_numpy(V).cuda()
        else:
            dV = torch.from_numpy(V.view(np.int16)).cuda().view(torch.bfloat16)
        ref = oracle.gather(V, N, d_v, idx, w.astype(np.float64))
    return dV, idx, w, ref


def gpu_read(dV, idx, w, B, H, n, d_v, k, vdt, read_sms):
    cfg = pk.make_config(32, d_v, B, H, n, k, q_dtype=pk.PKM_BF16, value_dtype=DT[vdt])
    h = pk.pkm_create(cfg)
    try:
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_READ_SMS, read_sms), "set_option")
        out = torch.full((B, d_v), float("nan"), device="cuda")
        pk.check(pk.pkm_gather(h, dV, B, H, n, k, torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w).cuda(), out), "pkm_gather")
        status = pk.pkm_get_status(h)
        return out.cpu().numpy().astype(np.float64), status
    finally:
        pk.pkm_destroy(h)


SHAPES = [
    # B, H, n, d_v, k, table dtype
    (50, 3, 16, 512, 7, "bf16"),    # 1 KB rows, 8 teams; bags of 21 rows (batches 8, 8, 5)
    (3, 1, 16, 1024, 5, "bf16"),    # fewer bags than a CTA's teams; a bag shorter than a batch
    (257, 4, 32, 1024, 32, "bf16"),  # the page row (2 KB) and bag (128 rows)
    (100, 2, 16, 256, 9, "f32"),    # fp32 rows of 1 KB, bags of 18 rows
    (64, 2, 16, 1024, 16, "fp8"),   # fp8 rows (1 KB of codes) with their row scales
    (33, 2, 16, 4096, 4, "bf16"),   # 8 KB rows: one team per CTA
    (40, 1, 8, 64, 3, "bf16"),      # 128-byte rows: the one-CTA-per-query form
]


@pytest.mark.parametrize("read_sms", [0, 1, 5])
@pytest.mark.parametrize("shape", SHAPES)
def test_read_matches_oracle(shape, read_sms):
    B, H, n, d_v, k, vdt = shape
    dV, idx, w, ref = read_case(sum(shape[:5]), B, H, n, d_v, k, vdt)
    got, status = gpu_read(dV, idx, w, B, H, n, d_v, k, vdt, read_sms)
    assert status == pk.PKM_OK
    err = np.abs(got - ref) / (1 + np.abs(ref))
    assert err.max() <= 1e-5, (shape, read_sms, float(err.max()))


@pytest.mark.parametrize("vdt", ["bf16", "fp8"])
def test_read_out_of_range_rows_skipped(vdt):
    # An index outside the table contributes nothing and sets
    # PKM_ERR_BAD_INDEX; the rest of its bag is read as usual.
    B, H, n, d_v, k = 20, 2, 16, 1024, 6
    dV, idx, w, _ = read_case(11, B, H, n, d_v, k, vdt)
    idx[4, 1, 3] = n * n
    idx[9, 0, 0] = -7
    keep = np.ones_like(w)
    keep[4, 1, 3] = keep[9, 0, 0] = 0.0
    safe = np.where(keep > 0, idx, 0)
    if vdt == "fp8":
        V = synth.normal(11, 3, n * n * d_v, 1.0, dtype="bf16")
        codes, scales = oracle.quantize_fp8(V, n * n, d_v)
        ref = oracle.gather_fp8(codes, scales, n * n, d_v, safe, (w * keep).astype(np.float64))
    else:
        V = synth.normal(11, 3, n * n * d_v, 1.0, dtype=vdt)
        ref = oracle.gather(V, n * n, d_v, safe, (w * keep).astype(np.float64))
    for read_sms in (0, 2):
        got, status = gpu_read(dV, idx, w, B, H, n, d_v, k, vdt, read_sms)
        assert status == pk.PKM_ERR_BAD_INDEX
        err = np.abs(got - ref) / (1 + np.abs(ref))
        assert err.max() <= 1e-5, (vdt, read_sms, float(err.max()))


def test_read_sms_option_range():
    cfg = pk.make_config(32, 512, 8, 1, 16, 4, q_dtype=pk.PKM_BF16)
    h = pk.pkm_create(cfg)
    try:
        assert pk.pkm_set_option(h, pk.PKM_OPT_READ_SMS, -1) == pk.PKM_ERR_OPTION
        assert pk.pkm_set_option(h, pk.PKM_OPT_READ_SMS, 1.5) == pk.PKM_ERR_OPTION
        assert pk.pkm_set_option(h, pk.PKM_OPT_READ_SMS, 10 ** 6) == pk.PKM_ERR_OPTION
        assert pk.pkm_set_option(h, pk.PKM_OPT_READ_SMS, 0) == pk.PKM_OK
    finally:
        pk.pkm_destroy(h)

