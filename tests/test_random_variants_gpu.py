"""Seeded random cases of the variants against the fp64 oracle.

Each case draws a variant -- a sliding window, attention dropout or a packed
variable-length batch -- and its shape: the head dimension (any multiple of
8 up to 256, so the D = 64, D = 128 and wide kernels all take every variant),
the element type, the mask, grouped K/V heads, a ragged sequence length and
the variant's own parameters (window bounds including 0 and unbounded sides,
the drop probability and seed, sequence lengths including empty ones).  The
case runs through the binding on the GPU and is compared with the oracle's
definition of that variant within the parity tolerances (dropout: plus what
the 1 / (1 - p) scale adds to the rounding of P).  The draws are fixed by the
case index, so a failure names a reproducible case.
"""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference, attention_reference_varlen
from oracle.dropout import attention_reference_dropout

from gpu_common import abs_weights, assert_close, assert_dropout_close

pytestmark = pytest.mark.gpu

N_CASES = 36
VARIANTS = ("window", "dropout", "packed")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import attention_forward_fwd_gb300 as fa
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    fa.build()
    fa.library()
    fa.fa_device_status(clear=True)
    yield
    assert fa.fa_device_status(clear=True) == 0


def _case(i):
    rng = np.random.default_rng(12000 + i)
    variant = VARIANTS[i % 3]
    D = int(8 * rng.integers(1, 33))
    dtype = "f16" if rng.integers(2) else "bf16"
    causal = bool(rng.integers(2))
    H = int(rng.choice([1, 2, 3, 4]))
    H_kv = int(rng.choice([d for d in range(1, H + 1) if H % d == 0]))
    return rng, variant, D, dtype, causal, H, H_kv


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_variant(i):
    import torch
    import attention_forward_fwd_gb300 as fa
    rng, variant, D, dtype, causal, H, H_kv = _case(i)
    scale = D ** -0.5
    what = f"random {variant} case {i}: D{D} {dtype} causal={causal} H{H}/{H_kv}"
    if variant == "packed":
        lens = [int(x) for x in rng.integers(0, 700, size=int(rng.integers(2, 8)))]
        lens[int(rng.integers(len(lens)))] = int(rng.integers(1, 700))   # at least one row
        qb, kb, vb, cu = fa_inputs.make_varlen(lens, H, D, dtype, "normal", 300 + i, h_kv=H_kv)
        q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
        o, lse = fa.attention_forward_varlen(q, k, v, torch.from_numpy(cu).cuda(), max(lens),
                                             causal=causal, scale=scale)
        torch.cuda.synchronize()
        Oref, Lref = attention_reference_varlen(qb, kb, vb, cu, dtype, causal, scale)
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                     f"{what} lens={lens}")
        return
    B = int(rng.integers(1, 3))
    S = int(rng.choice([1, 63, 128, 129, 300, 511, 777, 1000]))
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 400 + i, h_kv=H_kv)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    if variant == "window":
        left = int(rng.choice([-1, 0, int(rng.integers(1, S + 1))]))
        right = int(rng.choice([0, int(rng.integers(1, S + 1))] + ([] if left == -1 else [-1])))
        o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale, window=(left, right))
        torch.cuda.synchronize()
        Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale, window=(left, right))
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                     f"{what} S{S} window=({left}, {right})")
        return
    p = float(rng.choice([0.05, 0.3, 0.6]))
    seed = int(rng.integers(0, 2 ** 63))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    Oref, Lref = attention_reference_dropout(qb, kb, vb, dtype, causal, scale, p, seed)
    A = abs_weights(qb, kb, vb, dtype, causal, scale, p, seed)
    assert_dropout_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, A, dtype,
                         f"{what} S{S} p={p}")
