"""GPU parity of local (sliding-window) attention (fa_fwd_local) against the
fp64 oracle: key j is kept for query i iff i - left <= j <= i + right
(-1: no bound), the causal mask capping the right bound at 0.  Tolerances as
in test_parity_gpu.py."""
import pytest

import fa_inputs
from oracle import attention_reference

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
    assert fa.fa_device_status(clear=False) == 0, "a device-side wait timed out"


def _window_case(B, H, H_kv, S, D, dtype, causal, window, dist="normal", seed=70):
    import torch
    import attention_forward_fwd_gb300 as fa
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, dist, seed, h_kv=H_kv)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=D ** -0.5, window=window)
    torch.cuda.synchronize()
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, D ** -0.5, window=window)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                 f"window {window} causal={causal} S{S} D{D}")


@pytest.mark.parametrize("window,causal", [
    ((0, 0), False), ((0, 0), True), ((1, -1), True), ((37, -1), True), ((127, -1), True),
    ((128, -1), True), ((255, 0), False), ((200, 100), False), ((-1, 64), False),
    ((128, 128), False), ((513, -1), True),
])
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16")])
def test_windows(window, causal, D, dtype):
    _window_case(2, 4, 2, 1000, D, dtype, causal, window)


@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "f16")])
def test_window_many_items_and_peaky_scores(D, dtype):
    """Long sequence, narrow window: thousands of small work items, each
    query tile with its own start in the key ring; peaky scores."""
    _window_case(2, 16, 4, 4096, D, dtype, True, (300, -1), dist="stress", seed=71)


def test_covering_window_equals_the_unwindowed_call():
    import torch
    import attention_forward_fwd_gb300 as fa
    qb, kb, vb = fa_inputs.make_qkv(1, 4, 700, 64, "f16", "normal", 72)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    for causal in (False, True):
        o1, l1 = fa.attention_forward(q, k, v, causal=causal, split_kv=False)
        o2, l2 = fa.attention_forward(q, k, v, causal=causal, window=(700, 700))
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
