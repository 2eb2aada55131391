"""GPU parity on long sequences, against the fp64 oracle row by row.

Sequences of 32768 to 131077 rows (ragged ends included) for each kernel:
D = 64 and D = 128 with two query heads sharing one K/V head, and the wide
kernel at D = 256.  Every query block's key loop runs through hundreds of
key tiles (the K / V ring wraps many times within one work item), the split
planner sees shapes it splits and shapes with more query blocks than it ever
splits, and row offsets reach 2^17.  The first and the last 96 rows and
sampled rows of every head are compared with the oracle's plain definition,
which takes every one of the S keys for each of those rows; tolerances as
in test_parity_gpu.py.
"""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_rows

from gpu_common import assert_close, run_gpu

pytestmark = pytest.mark.gpu


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


def _rows(S, rng, n=24):
    # 96 rows at each end (the whole ragged last tile of every case here)
    edge = set(range(min(96, S))) | set(range(max(0, S - 96), S))
    fixed = {127, 128, 255, 256, 257, S // 2, S // 2 + 1, S - 129, S - 128}
    rnd = set(rng.integers(0, S, size=n).tolist())
    return sorted(r for r in edge | fixed | rnd if 0 <= r < S)


CASES = [
    # (S, D, dtype, H, H_kv)
    (32768, 64, "f16", 2, 1),
    (65613, 64, "f16", 2, 1),
    (131077, 64, "f16", 1, 1),
    (32768, 128, "bf16", 2, 1),
    (65613, 128, "bf16", 2, 1),
    (40000, 256, "bf16", 1, 1),
]


@pytest.mark.parametrize("S,D,dtype,H,H_kv", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_rows(S, D, dtype, H, H_kv, causal):
    scale = D ** -0.5
    seed = 700 + S % 97 + D + int(causal)
    qb, kb, vb = fa_inputs.make_qkv(1, H, S, D, dtype, "normal", seed, h_kv=H_kv)
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    rng = np.random.default_rng(seed)
    for h in range(H):
        rows = _rows(S, rng)
        Oref, Lref = attention_rows(qb, kb, vb, dtype, causal, scale, 0, h, rows)
        assert_close(O[0, rows, h, :], L[0, h, rows], Oref, Lref, dtype,
                     f"S{S} D{D} {dtype} H{H}/{H_kv} causal={causal} h{h}")
