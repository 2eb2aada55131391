"""fa_fwd_splitkv_static: the split-over-keys path with its scratch in a
device array inside the library, for callers that cannot allocate device
memory themselves (for example a latency-critical loop that must not pay for
cudaMalloc's implicit synchronisation, or code whose device memory belongs to
an allocator it cannot reach).

The tests call the entry point through the C-ABI and compare its output
with fa_fwd_splitkv (caller-provided workspace) and with the fp64 oracle on
the same inputs, within the parity tolerances: two calls in a row with
different inputs (the second call runs on the scratch the first one left
behind), and three calls queued back to back on one stream with no wait
between them (each call's main kernel may start while the previous call's
merge still reads the array).  They are collected last so that a failure
here stops a `-x` run only after every other test.
"""
import ctypes

import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference

from gpu_common import lse_tol, o_tol

pytestmark = pytest.mark.gpu

STATIC_BYTES = 24 << 20


@pytest.fixture(scope="module")
def lib():
    import torch
    import attention_forward_fwd_gb300 as fa
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    fa.build()
    lib = fa.library()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_splitkv_static.restype = i
    return lib


def _inputs(B, H, S, D, dtype, seed):
    """Device tensors and the 16-bit host bits they hold (for the oracle)."""
    bits = fa_inputs.make_qkv(B, H, S, D, dtype, "stress", seed)
    return tuple(fa_inputs.to_torch(x, dtype).cuda() for x in bits), bits


def _check(o, lse, o_ref, l_ref, bits, dtype, causal, scale, what):
    """o, lse against the caller-workspace result and against the oracle."""
    O, Oref = o.double().cpu().numpy(), o_ref.double().cpu().numpy()
    L, Lref = lse.double().cpu().numpy(), l_ref.double().cpu().numpy()
    assert np.all(np.abs(O - Oref) <= o_tol(Oref, dtype)), f"{what}: O differs from fa_fwd_splitkv"
    assert np.all(np.abs(L - Lref) <= lse_tol(Lref)), f"{what}: LSE differs from fa_fwd_splitkv"
    Oo, Lo = attention_reference(*bits, dtype, causal, scale)
    assert np.all(np.abs(O - Oo) <= o_tol(Oo, dtype)), f"{what}: O differs from the oracle"
    assert np.all(np.abs(L - Lo) <= lse_tol(Lo)), f"{what}: LSE differs from the oracle"


def _with_workspace(q, k, v, causal, scale, code):
    import torch
    import attention_forward_fwd_gb300 as fa
    B, S, H, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device)
    n = fa.fa_splitkv_workspace_size(B, H, S, D, causal)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    st = torch.cuda.current_stream().cuda_stream
    rc = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, S, D, causal, scale, code, ws.data_ptr(),
                           ws.numel(), st)
    assert rc == fa.FA_OK
    return o, lse


def _static(lib, q, k, v, causal, scale, code):
    import torch
    B, S, H, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device)
    rc = lib.fa_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, S, D, int(causal), scale, code,
                                   torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


@pytest.mark.parametrize("B,H,S,D,dtype,causal", [
    (1, 1, 4096, 64, "f16", False),
    (1, 1, 4096, 64, "f16", True),
    (1, 2, 2000, 128, "bf16", True),
    (2, 3, 300, 64, "f16", False),
    (1, 1, 3000, 40, "f16", True),      # other head dimensions: split on the D = 64 kernel
    (1, 1, 1500, 96, "bf16", False),    # ... on the D = 128 kernel
    (1, 2, 700, 256, "f16", True),      # D > 128: never split, no scratch
])
def test_static_scratch_matches_caller_workspace(lib, B, H, S, D, dtype, causal):
    import torch
    import attention_forward_fwd_gb300 as fa
    assert fa.fa_splitkv_workspace_size(B, H, S, D, causal) <= STATIC_BYTES
    code = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    scale = D ** -0.5
    for call, seed in enumerate((101, 202)):     # two calls in a row
        (q, k, v), bits = _inputs(B, H, S, D, dtype, seed + S)
        o_ref, l_ref = _with_workspace(q, k, v, causal, scale, code)
        rc, o, lse = _static(lib, q, k, v, causal, scale, code)
        assert rc == fa.FA_OK, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        _check(o, lse, o_ref, l_ref, bits, dtype, causal, scale, f"call {call}")
    assert fa.fa_device_status(clear=False) == fa.FA_OK


@pytest.mark.parametrize("B,H,S,D,dtype,causal", [
    (1, 1, 3000, 40, "f16", True),      # some query tiles see no key of a split
    (1, 1, 4096, 64, "f16", False),
])
def test_static_calls_back_to_back(lib, B, H, S, D, dtype, causal):
    """Three static calls with different inputs queued on one stream with no
    wait between them, then one synchronisation: each result must be that
    call's own (a call's merge must finish reading the shared array before
    the next call's main kernel writes it)."""
    import torch
    import attention_forward_fwd_gb300 as fa
    assert fa.fa_splitkv_launches(B, H, S, D, causal) == 2   # the split path runs
    code = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    scale = D ** -0.5
    cases = [_inputs(B, H, S, D, dtype, seed) for seed in (303, 404, 505)]
    refs = [_with_workspace(*qkv, causal, scale, code) for qkv, _ in cases]
    torch.cuda.synchronize()
    outs = []
    for qkv, _ in cases:
        rc, o, lse = _static(lib, *qkv, causal, scale, code)
        assert rc == fa.FA_OK, rc
        outs.append((o, lse))
    torch.cuda.synchronize()
    for n, ((o, lse), (o_ref, l_ref), (_, bits)) in enumerate(zip(outs, refs, cases)):
        _check(o, lse, o_ref, l_ref, bits, dtype, causal, scale, f"queued call {n}")
    assert fa.fa_device_status(clear=False) == fa.FA_OK


def test_static_scratch_rejects_shapes_beyond_its_size(lib):
    import torch
    import attention_forward_fwd_gb300 as fa
    # a block-starved shape whose split needs more than the static array
    B, H, S, D = 1, 1, 4096, 128
    assert fa.fa_splitkv_workspace_size(B, H, S, D, True) > STATIC_BYTES
    q = torch.zeros(B, S, H, D, dtype=torch.bfloat16, device="cuda")
    rc, _, _ = _static(lib, q, q, q, True, D ** -0.5, fa.FA_BF16)
    assert rc == fa.FA_ERR_UNSUPPORTED
