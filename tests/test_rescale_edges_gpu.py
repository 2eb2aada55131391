"""GPU parity at the edges of the lazy rescale.

The kernels keep a reference max per row and move it only when a key tile
would push some probability past 2^8 (D = 64: the tile max exceeds the
reference by more than 8 in log2 units; D >= 128: the tile's row sum against
the old reference exceeds 2^8, then the max is taken).  Until it moves, P
holds values up to 2^8 rather than at most 1.  These inputs sit on both sides
of that threshold:

* query rows and key tiles of mixed norms (row to row within one warp, tile
  to tile along the keys), so that some rows of a warp move their reference
  on a tile and others do not;
* every query row one vector q0 and single keys aligned with it, whose scores
  lie m + 7.9, m + 8.1 and m + 17 (log2 units) above the reference m set by
  the first key tile: just inside the threshold, just past it, and far past.

Each case is compared with the fp64 oracle element by element, tolerances as
in test_parity_gpu.py.
"""
import math

import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference, decode

from gpu_common import assert_close, run_gpu

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


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


def _mixed(dtype, seed, D, B=2, H=3, S=1100):
    """Q, K ~ N(0,1) with each query row scaled by one of 0.25 .. 2.5 (the
    factor changes from row to row) and each key tile of 128 by one of
    0.3 .. 3; V ~ U[-1, 1] as in the stress workload (the rows with large
    norms have a peaked softmax, where a 16-bit P's rounding times |v| is
    the error budget)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, S, H, D), dtype=np.float32)
    k = rng.standard_normal((B, S, H, D), dtype=np.float32)
    v = rng.uniform(-1.0, 1.0, size=(B, S, H, D)).astype(np.float32)
    row_f = np.array([0.25, 1.0, 0.6, 2.5, 1.0, 1.5, 0.8, 1.0], dtype=np.float32)
    tile_f = np.array([1.0, 0.3, 2.0, 1.0, 3.0, 0.5, 1.0, 1.2, 2.5], dtype=np.float32)
    q *= row_f[(np.arange(S) * 7 // 3) % len(row_f)][None, :, None, None]
    k *= tile_f[(np.arange(S) // 128) % len(tile_f)][None, :, None, None]
    return tuple(fa_inputs.f32_to_bits(x, dtype) for x in (q, k, v))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("split", [False, True])
def test_mixed_norms(D, dtype, causal, split):
    scale = 1.0 / math.sqrt(D)
    qb, kb, vb = _mixed(dtype, 71 + 2 * causal + 4 * split + (dtype == "bf16") + D, D)
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale, split_kv=split)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale)
    assert_close(O, L, Oref, Lref, dtype, f"mixed norms D{D} {dtype} causal={causal} split={split}")


# (key index, score above the reference in log2 units)
ALIGNED = ((2 * 128 + 37, 7.9), (3 * 128 + 5, 8.1), (5 * 128 + 90, 17.0))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_aligned_keys(D, dtype):
    """Every query row is one vector q0; keys are 0.5 N(0,1) except the
    aligned keys beta * q0 of ALIGNED, placed per head from the reference
    max m that key tile 0 sets (the other tiles' random keys stay below it
    plus 4).  Non-causal, so every row sees the same keys."""
    B, H, S = 1, 2, 1024
    scale = 1.0 / math.sqrt(D)
    c = scale * LOG2E
    rng = np.random.default_rng(404 + (dtype == "bf16") + D)
    q0 = rng.standard_normal(D).astype(np.float32)
    q = np.broadcast_to(q0, (B, S, H, D)).copy()
    k = 0.5 * rng.standard_normal((B, S, H, D)).astype(np.float32)
    v = rng.uniform(-1.0, 1.0, size=(B, S, H, D)).astype(np.float32)
    qb = fa_inputs.f32_to_bits(q, dtype)
    q0r = decode(qb, dtype)[0, 0, 0]                   # q0 as stored
    k0 = decode(fa_inputs.f32_to_bits(k, dtype), dtype)
    qq = float(q0r @ q0r)
    m_c = []
    for h in range(H):
        m_c.append(float((k0[0, :128, h] @ q0r).max()) * c)   # reference after tile 0, log2 units
        for idx, above in ALIGNED:
            k[0, idx, h, :] = ((m_c[h] + above) / (c * qq)) * q0
    kb = fa_inputs.f32_to_bits(k, dtype)
    vb = fa_inputs.f32_to_bits(v, dtype)
    kd = decode(kb, dtype)
    for h in range(H):
        for idx, above in ALIGNED:
            got = float(kd[0, idx, h] @ q0r) * c - m_c[h]
            assert abs(got - above) < 0.08, f"aligned key {idx} of head {h} lands {got:.3f} above m"
        # the random keys of the later tiles stay below the first tile's max plus 4
        assert float((k0[0, 128:, h] @ q0r).max()) * c < m_c[h] + 4.0
    for split in (False, True):
        O, L = run_gpu(qb, kb, vb, dtype, False, scale, split_kv=split)
        Oref, Lref = attention_reference(qb, kb, vb, dtype, False, scale)
        assert_close(O, L, Oref, Lref, dtype, f"aligned keys D{D} {dtype} split={split}")
