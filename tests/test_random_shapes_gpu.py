"""Seeded random shapes against the fp64 oracle, element by element.

Each case draws the batch, the query heads and a K/V head count dividing
them, a sequence length (often not a multiple of any tile), a head dimension
(any multiple of 8 up to 256, so every kernel width and the zero-padded
columns are reached), the mask, the element type, the input distribution and
whether the keys may be split over CTAs; the case runs through the binding
on the GPU and is compared with the plain fp64 definition within the parity
tolerances.  The draws are fixed by the case index, so a failure names a
reproducible shape.
"""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference

from gpu_common import assert_close, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 48


def _case(i):
    rng = np.random.default_rng(9000 + i)
    B = int(rng.integers(1, 4))
    H = int(rng.choice([1, 2, 3, 4, 6, 8]))
    H_kv = int(rng.choice([d for d in range(1, H + 1) if H % d == 0]))
    S = int(rng.choice([1, 7, 64, 127, 128, 129, 255, 256, 257, 300, 511, 640, 777, 1000]))
    D = int(8 * rng.integers(1, 33))
    causal = bool(rng.integers(2))
    dtype = "f16" if rng.integers(2) else "bf16"
    dist = "stress" if rng.integers(4) == 0 else "normal"
    split = bool(rng.integers(2))
    return B, H, H_kv, S, D, causal, dtype, dist, split


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    B, H, H_kv, S, D, causal, dtype, dist, split = _case(i)
    scale = D ** -0.5
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, dist, 500 + i, h_kv=H_kv)
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale, split_kv=split)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale)
    assert_close(O, L, Oref, Lref, dtype,
                 f"random case {i}: B{B} H{H} Hkv{H_kv} S{S} D{D} causal={causal} {dtype} {dist} split={split}")
