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
