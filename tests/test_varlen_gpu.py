"""GPU parity of the packed variable-length batch (fa_fwd_varlen) against the
fp64 oracle: sequence b is rows cu[b] .. cu[b+1]-1 and attends within itself.
Tolerances as in test_parity_gpu.py."""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference_varlen

from gpu_common import assert_close

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
    assert fa.fa_device_status(clear=False) == 0, "a device-side check failed"


def _run(qb, kb, vb, cu, dtype, causal, scale, max_seqlen=None):
    import torch
    import attention_forward_fwd_gb300 as fa
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    cu_t = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    ms = int(np.diff(cu).max()) if max_seqlen is None else max_seqlen
    o, lse = fa.attention_forward_varlen(q, k, v, cu_t, max(ms, 1), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


EDGE = [1, 127, 128, 129, 255, 256, 257, 0, 300, 513, 1000, 2]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,H_kv,D,dtype", [(4, 2, 64, "f16"), (4, 4, 128, "bf16"), (6, 1, 64, "bf16"),
                                            (2, 2, 128, "f16")])
def test_varlen_edge_lengths(H, H_kv, D, dtype, causal):
    qb, kb, vb, cu = fa_inputs.make_varlen(EDGE, H, D, dtype, "normal", 60 + H + D, h_kv=H_kv)
    O, L = _run(qb, kb, vb, cu, dtype, causal, D ** -0.5)
    Oref, Lref = attention_reference_varlen(qb, kb, vb, cu, dtype, causal, D ** -0.5)
    assert_close(O, L, Oref, Lref, dtype, f"varlen H{H}/{H_kv} D{D} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_many_sequences(causal):
    """64 sequences of 1..700 rows, 8 heads: many items per CTA, most CTAs
    meet items past a sequence's end (skipped)."""
    lens = fa_inputs.varlen_lengths(64, 1, 700, 61)
    qb, kb, vb, cu = fa_inputs.make_varlen(lens, 8, 64, "f16", "stress", 62, h_kv=4)
    O, L = _run(qb, kb, vb, cu, "f16", causal, 0.125)
    Oref, Lref = attention_reference_varlen(qb, kb, vb, cu, "f16", causal, 0.125)
    assert_close(O, L, Oref, Lref, "f16", f"varlen x64 causal={causal}")


@pytest.mark.parametrize("S,D,dtype", [(300, 64, "f16"), (512, 128, "bf16")])
def test_varlen_equal_lengths_match_the_batched_call_bitwise(S, D, dtype):
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H = 3, 4
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 63)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    for causal in (False, True):
        o, lse = fa.attention_forward(q, k, v, causal=causal, split_kv=False)
        cu = torch.arange(B + 1, dtype=torch.int32, device="cuda") * S
        ov, lv = fa.attention_forward_varlen(q.view(B * S, H, D), k.view(B * S, H, D),
                                             v.view(B * S, H, D), cu, S, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(ov.view(B, S, H, D), o)
        assert torch.equal(lv.view(H, B, S).permute(1, 0, 2), lse)


@pytest.mark.parametrize("D", [64, 256])
def test_varlen_bad_offsets_are_reported_and_nothing_is_written_outside(D):
    """A sequence reaching past the packed tensors, and one longer than
    max_seqlen, are skipped and reported; the rest is computed, nothing is
    written outside the tensors (guard bands), the skipped rows keep their
    previous contents (D = 256: the wide kernel)."""
    import torch
    import attention_forward_fwd_gb300 as fa
    H, total = 2, 400
    qb, kb, vb, _ = fa_inputs.make_varlen([total], H, D, "f16", "normal", 64)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    guard = 4096
    for cu_list, ms in (([0, 100, 5000], 300), ([0, 100, 400], 200)):
        buf = torch.full((total * H * D + 2 * guard,), 7.0, dtype=torch.float16, device="cuda")
        o = buf[guard:guard + total * H * D].view(total, H, D)
        lbuf = torch.full((H * total + 2 * 64,), 3.0, dtype=torch.float32, device="cuda")
        lse = lbuf[64:64 + H * total].view(H, total)
        cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
        fa.fa_device_status(clear=True)
        fa.attention_forward_varlen(q, k, v, cu, ms, causal=True, scale=D ** -0.5, out=o, lse=lse)
        assert fa.fa_device_status(clear=True) == fa.FA_ERR_BAD_SEQLENS
        assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + total * H * D:] == 7.0)
        assert torch.all(lbuf[:64] == 3.0) and torch.all(lbuf[64 + H * total:] == 3.0)
        assert torch.all(o[100:] == 7.0) and torch.all(lse[:, 100:] == 3.0)
        good = np.array([0, 100], dtype=np.int32)
        Oref, Lref = attention_reference_varlen(qb[:100], kb[:100], vb[:100], good, "f16", True, D ** -0.5)
        assert_close(o[:100].double().cpu().numpy(), lse[:, :100].double().cpu().numpy(), Oref, Lref,
                     "f16", f"varlen good part D{D}")
