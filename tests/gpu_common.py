"""Helpers shared by the GPU parity tests (not collected by pytest)."""
import numpy as np

import fa_inputs

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
