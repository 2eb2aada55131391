"""The bounded waits end a kernel whose input never arrives in a timeout
status instead of a hang, and the CUDA context stays usable.  The test
support call withholds the first query tile's load; no GPU fault is made.
(Collected late: it leaves a device status behind until it clears it.)"""
import time

import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference

from gpu_common import assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.timeout(120)
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (128, "f16"), (64, "bf16"),
                                     (256, "bf16"), (256, "f16"), (192, "bf16")])   # the wide kernel too
def test_withheld_load_ends_in_timeout_not_a_hang(D, dtype):
    import torch
    import attention_forward_fwd_gb300 as fa
    fa.build()
    fa.fa_device_status(clear=True)
    S = 512
    q = torch.zeros(1, S, 1, D, dtype=torch.float16 if dtype == "f16" else torch.bfloat16,
                    device="cuda")
    o = torch.empty_like(q)
    code = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    t0 = time.time()
    rc = fa.library().fa_selftest_timeout(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                                          S, D, code, None)
    assert rc == fa.FA_OK
    # the stream-ordered read sees the timeout once the call's work is done
    # (and does not clear it); the device-wide read then clears it
    assert fa.fa_last_device_status(None) == fa.FA_ERR_TIMEOUT
    status = fa.fa_device_status(clear=True)
    elapsed = time.time() - t0
    assert status == fa.FA_ERR_TIMEOUT, status
    assert fa.fa_last_device_status(None) == fa.FA_OK
    assert elapsed < 30.0, elapsed                      # seconds, not a hang
    assert fa.fa_device_status(clear=False) == fa.FA_OK
    # the context is still usable: a normal call afterwards is exact
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 300, D, dtype, "normal", 80)
    O, L = run_gpu(qb, kb, vb, dtype, True, D ** -0.5)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, True, D ** -0.5)
    assert_close(O, L, Oref, Lref, dtype, "after the timeout")
    assert fa.fa_device_status(clear=False) == fa.FA_OK


def test_last_device_status_on_a_side_stream():
    """An ordinary call on a torch side stream leaves the status word at
    FA_OK, read in that stream's order."""
    import torch
    import attention_forward_fwd_gb300 as fa
    fa.build()
    fa.fa_device_status(clear=True)
    side = torch.cuda.Stream()
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 500, 64, "f16", "normal", 81)
    O, L = run_gpu(qb, kb, vb, "f16", False, 0.125, stream=side)
    assert fa.fa_last_device_status(side) == fa.FA_OK
    Oref, Lref = attention_reference(qb, kb, vb, "f16", False, 0.125)
    assert_close(O, L, Oref, Lref, "f16", "side stream")
