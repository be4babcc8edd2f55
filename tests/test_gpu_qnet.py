"""The query network on the GPU against the fp64 oracle.

Product-Key Memory, code listing: q = BatchNorm1d(Linear(dim, F, bias=False)(x)),
here with the BatchNorm's running statistics.  The GPU path folds the
BatchNorm into a per-feature scale and shift (pkm_bn_fold) and multiplies on
the tensor cores with fp32 accumulation (pkm_query_net); q is bf16.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pk = pytest.importorskip("sparse_top_lookup_gb300")


def dev16(a):
    return torch.from_numpy(a.view(np.int16)).cuda()


def run_gpu(x, W, B, dim, F, gamma, beta, mean, var, eps):
    t = [torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
         for a in (gamma, beta, mean, var)]
    scale = torch.empty(F, device="cuda")
    shift = torch.empty(F, device="cuda")
    pk.check(pk.pkm_bn_fold(*t, eps, F, scale, shift), "bn_fold")
    q = torch.empty(B, F, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.check(pk.pkm_query_net(dev16(x), dev16(W), B, dim, F, scale, shift, q, status), "qnet")
    torch.cuda.synchronize()
    assert status.item() == pk.PKM_OK
    return (q.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)


def bn_params(rng, F):
    gamma = (1 + 0.2 * rng.standard_normal(F)).astype(np.float32)
    beta = (0.3 * rng.standard_normal(F)).astype(np.float32)
    mean = (0.1 * rng.standard_normal(F)).astype(np.float32)
    var = (0.5 + rng.random(F)).astype(np.float32)
    return gamma, beta, mean, var


@pytest.mark.parametrize("B,dim,F", [(300, 1024, 4096), (129, 48, 96), (64, 256, 288),
                                     (1000, 512, 512)])
def test_query_net_matches_oracle(B, dim, F):
    rng = np.random.default_rng(B + dim + F)
    x = synth.normal(B, 6, B * dim, 1.0, dtype="bf16").reshape(B, dim)
    W = synth.normal(B, 7, F * dim, 1.0 / dim, dtype="bf16").reshape(F, dim)
    gamma, beta, mean, var = bn_params(rng, F)
    eps = 1e-5
    got = run_gpu(x, W, B, dim, F, gamma, beta, mean, var, eps)
    ref = oracle.query_net(x, W, B, dim, F, gamma, beta, mean, var, eps)
    # bf16 rounding of the output (half an ulp: at most 2^-8 of the value, at
    # the bottom of a binade) plus the fp32 accumulation and fold error,
    # bounded by dim * 2^-24 of sum_t |x W| * |scale|
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.abs(gamma / np.sqrt(var.astype(np.float64) + eps))
    acc = (np.abs(xf) @ np.abs(wf).T) * scale + np.abs(mean) * scale + np.abs(beta)
    tol = 2.0 ** -8 * np.abs(ref) * (1 + 1e-6) + (dim + 8) * 2.0 ** -24 * acc * 1.01
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])


def test_query_net_integer_inputs_exact():
    # integer x and W are exact in bf16 and their products sum exactly in fp32;
    # with scale 1 and shift 0 (var + eps = 1) every output is an integer below
    # 256, exact in bf16: any indexing slip of the tiles shows bit for bit
    rng = np.random.default_rng(33)
    B, dim, F = 257, 96, 544
    xi = rng.integers(-2, 3, (B, dim)).astype(np.float32)
    wi = rng.integers(-1, 2, (F, dim)).astype(np.float32)
    x = synth_bf16(xi)
    W = synth_bf16(wi)
    one, zero = np.ones(F, np.float32), np.zeros(F, np.float32)
    got = run_gpu(x, W, B, dim, F, one, zero, zero, np.full(F, 0.75, np.float32), 0.25)
    want = xi.astype(np.float64) @ wi.astype(np.float64).T
    assert np.abs(want).max() < 256
    assert (got == want).all()


def synth_bf16(a):
    # exact: these values are small integers
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- training form
#
# Product-Key Memory, "Keeping the memory in use": the queries' BatchNorm with
# the batch's own statistics (pkm_query_net_batch).

def run_gpu_batch(x, W, B, dim, F, gamma, beta, eps):
    g, bt = (torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda() for a in (gamma, beta))
    ws = torch.empty(max(pk.pkm_query_net_batch_workspace_bytes(B, F), 16), dtype=torch.uint8,
                     device="cuda")
    q = torch.empty(B, F, dtype=torch.int16, device="cuda")
    mean = torch.empty(F, device="cuda")
    var = torch.empty(F, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.check(pk.pkm_query_net_batch(dev16(x), dev16(W), B, dim, F, g, bt, eps, ws, q, mean, var,
                                    status), "qnet_batch")
    torch.cuda.synchronize()
    assert status.item() == pk.PKM_OK
    qf = (q.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return qf, mean.cpu().numpy(), var.cpu().numpy()


def check_batch(x, W, B, dim, F, gamma, beta, eps):
    got, gm, gv = run_gpu_batch(x, W, B, dim, F, gamma, beta, eps)
    ref, rm, rv = oracle.query_net_batch(x, W, B, dim, F, gamma, beta, eps)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    z = xf @ wf.T
    acc = np.abs(xf) @ np.abs(wf).T  # bound on the fp32 accumulation error, / 2^-24 / dim
    rms = np.sqrt((z ** 2).mean(0))
    s = np.abs(gamma) / np.sqrt(rv + eps)
    # statistics: fp32 block sums (32 rows) combined in fp64 and the fp32
    # accumulation of z, relative ~2^-19 of the feature's rms
    zerr = (dim + 8) * 2.0 ** -24 * acc.max(0)
    assert (np.abs(gm - rm) <= 2.0 ** -17 * rms + zerr).all()
    assert (np.abs(gv - rv) <= 2.0 ** -16 * rv + 2 * rms * zerr + 1e-30).all()
    # q: bf16 rounding (at most 2^-8 of the value) + z's accumulation error
    # and the statistics' error, both through the scale
    tol = (2.0 ** -8 * np.abs(ref) * (1 + 1e-6) + s * (dim + 8) * 2.0 ** -24 * acc * 1.01
           + 2.0 ** -15 * (np.abs(ref - beta) + s * (rms + zerr)))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    return got, ref


@pytest.mark.parametrize("B,dim,F", [(300, 1024, 4096), (129, 48, 96), (64, 256, 288),
                                     (1000, 512, 512), (33, 64, 96), (2, 32, 64),
                                     (4096, 512, 1024)])
def test_query_net_batch_matches_oracle(B, dim, F):
    rng = np.random.default_rng(B * 7 + dim + F)
    x = synth.normal(B + 1, 6, B * dim, 1.0, dtype="bf16").reshape(B, dim)
    W = synth.normal(B + 1, 7, F * dim, 1.0 / dim, dtype="bf16").reshape(F, dim)
    gamma, beta, _, _ = bn_params(rng, F)
    got, _ = check_batch(x, W, B, dim, F, gamma, beta, 1e-5)
    # the batch's own statistics: every feature leaves with mean ~beta
    if B >= 64:
        assert (np.abs(got.mean(0) - beta) < 0.05).all()


def test_query_net_batch_offset_features_and_single_row():
    # a large common offset in one input column: every feature's mean is far
    # above its spread (the variance must not come from a difference of
    # large sums); then B = 1, where the variance is 0 and q = beta
    rng = np.random.default_rng(44)
    B, dim, F = 257, 64, 128
    xf = rng.standard_normal((B, dim)).astype(np.float32)
    xf[:, 3] = 64.0 + xf[:, 3] / 64
    x = synth.f32_to_bf16(xf)
    W = synth.normal(9, 7, F * dim, 1.0 / dim, dtype="bf16").reshape(F, dim)
    gamma, beta, _, _ = bn_params(rng, F)
    check_batch(x, W, B, dim, F, gamma, beta, 1e-5)
    got, _, gv = run_gpu_batch(x[:1], W, 1, dim, F, gamma, beta, 1e-3)
    assert (gv == 0).all()
    # z * s + t with t = beta - z * s: beta up to the fp32 rounding of s and
    # t (relative 2^-24 of |z s|), then bf16
    np.testing.assert_allclose(got[0], beta, rtol=2.0 ** -8, atol=1e-4)


def test_query_net_batch_argument_errors():
    x = torch.zeros(4, 32, dtype=torch.int16, device="cuda")
    W = torch.zeros(64, 32, dtype=torch.int16, device="cuda")
    g = torch.ones(64, device="cuda")
    ws = torch.empty(pk.pkm_query_net_batch_workspace_bytes(4, 64), dtype=torch.uint8,
                     device="cuda")
    q = torch.empty(4, 64, dtype=torch.int16, device="cuda")
    assert pk.pkm_query_net_batch(x, W, 0, 32, 64, g, g, 1e-5, ws, q) == pk.PKM_OK
    assert pk.pkm_query_net_batch(x, W, 4, 32, 64, g, g, -1.0, ws, q) == pk.PKM_ERR_INVALID
    assert pk.pkm_query_net_batch(x, W, 4, 32, 48, g, g, 1e-5, ws, q) == pk.PKM_ERR_UNSUPPORTED
    assert pk.pkm_query_net_batch(x, W, 4, 32, 64, g, g, 1e-5, None, q) == pk.PKM_ERR_INVALID
    assert pk.pkm_query_net_batch_workspace_bytes(-1, 64) == 0
