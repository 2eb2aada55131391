"""Helpers shared by the GPU parity tests (not collected by pytest)."""
import numpy as np

import fa_inputs
from oracle import dropout_keep
from oracle.attention import decode

TOL_O = {"f16": 2e-3, "bf16": 8e-3}


def lse_tol(ref_lse):
    return 1e-4 * np.abs(ref_lse) + 1e-4


def run_gpu(qb, kb, vb, dtype, causal, scale, with_lse=True, stream=None, split_kv=True):
    """Copy 16-bit inputs to cuda:0, run the library, return (O f64, LSE f64)."""
    import torch
    import attention_forward_fwd_gb300 as fa
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # the uploads land first
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale, with_lse=with_lse,
                                  stream=stream, split_kv=split_kv)
    torch.cuda.synchronize()
    O = o.double().cpu().numpy()
    L = lse.double().cpu().numpy() if lse is not None else None
    return O, L


# significant bits of the 16-bit output types
_PREC = {"f16": 11, "bf16": 8}
_EMIN = {"f16": -14, "bf16": -126}


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit output type at |x|: the error that the
    final rounding of O to its storage type may add on its own."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** _EMIN[dtype])))
    return 0.5 * np.exp2(e - (_PREC[dtype] - 1))


def o_tol(Oref, dtype):
    """max|dO| bound: the stated tolerance on the result, plus the half ulp
    of the 16-bit type that O is stored in."""
    return TOL_O[dtype] + half_ulp(Oref, dtype)


# (what, max|dO|, largest share of its bound used, max|dLSE|, share used) of
# every comparison in this process; the terminal summary reports them
MARGINS = []


def assert_close(O, L, Oref, Lref, dtype, what=""):
    dO = np.abs(O - Oref)
    assert np.all(np.isfinite(O)), f"{what}: non-finite O"
    tol = o_tol(Oref, dtype)
    bad = dO > tol
    assert not bad.any(), f"{what}: max|dO| = {dO.max():.3e} at {np.unravel_index(dO.argmax(), dO.shape)}"
    rec = [what, float(dO.max()), float((dO / tol).max()), None, None]
    if L is not None:
        dL = np.abs(L - Lref)
        ltol = lse_tol(Lref)
        bad = dL > ltol
        assert not bad.any(), f"{what}: |dLSE| = {dL.max():.3e} at {np.unravel_index(dL.argmax(), dL.shape)}"
        rec[3:] = [float(dL.max()), float((dL / ltol).max())]
    MARGINS.append(tuple(rec))


def assert_bare_tolerance(O, Oref, dtype, what=""):
    """The stated bound max|dO| <= 2e-3 (fp16) / 8e-3 (bf16) with no output
    rounding allowance, on the elements whose half ulp is below 1e-4 (there
    the rounding of O to 16 bits cannot account for any of the bound)."""
    sel = half_ulp(Oref, dtype) < 1e-4
    assert sel.any(), f"{what}: no element with a half ulp below 1e-4"
    dO = np.abs(O - Oref)[sel]
    assert dO.max() <= TOL_O[dtype], f"{what}: max|dO| = {dO.max():.3e} on {sel.sum()} small elements"


# Dropout: the kernel rounds each kept P_ij to 16 bits (unit roundoff U16)
# before the 1 / (1 - p) scale, so element (i, d) may move by up to
# U16 * sum_j keep_ij P_ij |V_jd| / (1 - p) on top of the forward's error
# (twice that is allowed, for the exponential's own error).
U16 = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def abs_weights(qb, kb, vb, dtype, causal, scale, p, seed):
    """A[b, i, h, d] = sum_j keep_bhij P_bhij |V_bjd| / (1 - p) in fp64 (the
    oracle's probabilities and mask): the size of the sum whose terms the
    16-bit rounding of P perturbs."""
    q, k, v = decode(qb, dtype), decode(kb, dtype), decode(vb, dtype)
    B, S, H, _ = q.shape
    group = H // k.shape[2]
    keep = dropout_keep(B, H, S, p, seed)
    A = np.empty(q.shape[:3] + (v.shape[3],))
    vis = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
    for b in range(B):
        for h in range(H):
            z = np.where(vis, scale * (q[b, :, h, :] @ k[b, :, h // group, :].T), -np.inf)
            e = np.exp(z - z.max(axis=1, keepdims=True))
            P = e / e.sum(axis=1, keepdims=True)
            A[b, :, h, :] = (P * keep[b, h]) @ np.abs(v[b, :, h // group, :]) / (1.0 - p)
    return A


def assert_dropout_close(O, L, Oref, Lref, A, dtype, what):
    assert np.all(np.isfinite(O)), f"{what}: non-finite O"
    dO = np.abs(O - Oref)
    bound = TOL_O[dtype] + half_ulp(Oref, dtype) + 2.0 * U16[dtype] * A
    bad = dO > bound
    assert not bad.any(), f"{what}: max|dO| = {dO.max():.3e} at {np.unravel_index(dO.argmax(), dO.shape)}"
    dL = np.abs(L - Lref)
    assert not (dL > lse_tol(Lref)).any(), f"{what}: |dLSE| = {dL.max():.3e}"
