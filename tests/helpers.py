"""Shared test helpers: device tensors from the seeded generator, the parity
rule (indices bit-exact outside near-ties, weights and outputs within
2e-3 * (1 + |ref|)), and handle creation through the C ABI."""
import numpy as np

import oracle
import synth

TOL = 2e-3          # |gpu - ref| <= TOL * (1 + |ref|)
NEAR_TIE = 1e-5     # relative score gap below which two keys may swap


def to_device(a, dtype):
    """numpy (float32 or uint16 bf16 bits) -> CUDA torch tensor of the same bits."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def widen(a, dtype):
    return a.astype(np.float64) if dtype == "f32" else synth.bf16_to_f32(a).astype(np.float64)


def exact_scores(q, C, dtype, H, d_q, n, flat):
    """fp64 score of each flat key in `flat` [B, H, k] (for judging near-ties)."""
    B = flat.shape[0]
    qd = widen(q, dtype).reshape(B, H, d_q)
    Cd = widen(C, dtype).reshape(H, 2, n, d_q // 2)
    a, b = flat // n, flat % n
    out = np.empty(flat.shape)
    for h in range(H):
        s1 = np.einsum("bt,bjt->bj", qd[:, h, : d_q // 2], Cd[h, 0][a[:, h]])
        s2 = np.einsum("bt,bjt->bj", qd[:, h, d_q // 2:], Cd[h, 1][b[:, h]])
        out[:, h] = s1 + s2
    return out


def compare_lookup(gidx, gw, ref, q=None, C=None, dtype=None, H=None, d_q=None, n=None):
    """Parity of one lookup.  Returns dict(mismatch, near_ties, failures, max_w_err).

    A (query, head) whose index list differs from the oracle's counts as a
    near-tie when every GPU-selected key's exact fp64 score is within
    NEAR_TIE (relative) of the oracle's score at the same position, i.e. the
    lists differ only by keys that score the same to 1e-5; otherwise it is a
    failure.
    """
    ridx, rw, rsc = ref["idx"], ref["w"], ref["score"]
    mism = ~(gidx == ridx).all(-1)
    near, fail = 0, 0
    if mism.any():
        gsc = exact_scores(q, C, dtype, H, d_q, n, gidx) if q is not None else None
        for b, h in zip(*np.nonzero(mism)):
            ok = False
            if gsc is not None and len(set(gidx[b, h].tolist())) == gidx.shape[-1]:
                den = np.maximum(np.abs(rsc[b, h]), 1e-30)
                ok = bool((np.abs(gsc[b, h] - rsc[b, h]) / den < NEAR_TIE).all())
            near += ok
            fail += not ok
    werr = np.abs(gw.astype(np.float64) - rw) / (1 + np.abs(rw))
    return dict(mismatch=int(mism.sum()), near_ties=near, failures=fail,
                max_w_err=float(werr.max()) if werr.size else 0.0, w_ok=bool((werr <= TOL).all()))


def compare_out(gout, values, N, d_v, gidx, ref_idx, ref_w, ref_out, regather=None):
    """Output parity; queries whose selection was a near-tie swap are judged
    against the fp64 read of the GPU's rows with the oracle's weights
    (`regather(idx, w)` replaces the plain read, e.g. for an fp8 table)."""
    ref = ref_out.copy()
    swapped = ~(gidx == ref_idx).all(-1).all(-1)
    if swapped.any():
        if regather is None:
            ref[swapped] = oracle.gather(values, N, d_v, gidx[swapped], ref_w[swapped])
        else:
            ref[swapped] = regather(gidx[swapped], ref_w[swapped])
    err = np.abs(gout.astype(np.float64) - ref) / (1 + np.abs(ref))
    return float(err.max()) if err.size else 0.0


def make_handle(cfgd, B=None, staging=False):
    import sparse_top_lookup_gb300 as pk
    dt = pk.PKM_F32 if cfgd["dtype"] == "f32" else pk.PKM_BF16
    cfg = pk.make_config(cfgd["d_q"], cfgd["d_v"], B or cfgd["B"], cfgd["H"], cfgd["n_keys"],
                         cfgd["k"], q_dtype=dt, host_staging=staging)
    return pk.pkm_create(cfg), cfg
