"""GPU parity of attention dropout (fa_fwd_dropout) against the fp64 oracle.

Every probability P_ij is kept iff its 16-bit Philox4x32-10 draw is >=
floor(p * 2^16) and the kept ones are scaled by 1 / (1 - p); LSE is the
undropped one.
The keep decision is an integer comparison, so the mask is checked bit for
bit (read back through a V that routes each key to its own output column).
O is checked element by element against the oracle within the forward's
tolerance plus what the 1 / (1 - p) scale adds to the rounding of P: the
kernel rounds each kept P_ij to 16 bits (relative error u, 2^-11 in fp16 and
2^-8 in bf16) before the scale, so element (i, d) may move by up to
u * sum_j keep_ij P_ij |V_jd| / (1 - p) on top of the forward's error
(twice that is allowed, for the exponential's own error).
"""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference_dropout, dropout_keep
from oracle.attention import decode

from gpu_common import abs_weights as _abs_weights, assert_dropout_close as _assert_dropout_close

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


def _run(qb, kb, vb, dtype, causal, scale, p, seed):
    import torch
    import attention_forward_fwd_gb300 as fa
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (256, "bf16"), (192, "f16")])
def test_dropout_matches_oracle(p, causal, D, dtype):
    """Several query and key tiles with a ragged tail, grouped K/V heads."""
    B, H, H_kv, S = 2, 4, 2, 333
    seed = 0x1234_5678_9ABC_DEF0
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 80, h_kv=H_kv)
    O, L = _run(qb, kb, vb, dtype, causal, D ** -0.5, p, seed)
    Oref, Lref = attention_reference_dropout(qb, kb, vb, dtype, causal, D ** -0.5, p, seed)
    A = _abs_weights(qb, kb, vb, dtype, causal, D ** -0.5, p, seed)
    _assert_dropout_close(O, L, Oref, Lref, A, dtype, f"p={p} causal={causal} D{D}")


@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (256, "bf16")])
def test_dropout_peaky_scores_several_items_per_cta(D, dtype):
    """More work items than SMs and peaky scores (the reference max moves)."""
    B, H, S = 3, 8, 1999
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "stress", 81)
    O, L = _run(qb, kb, vb, dtype, True, D ** -0.5, 0.2, 7)
    Oref, Lref = attention_reference_dropout(qb, kb, vb, dtype, True, D ** -0.5, 0.2, 7)
    A = _abs_weights(qb, kb, vb, dtype, True, D ** -0.5, 0.2, 7)
    _assert_dropout_close(O, L, Oref, Lref, A, dtype, f"stress D{D}")


@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (256, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_probability_is_the_plain_forward_bit_for_bit(D, dtype, causal):
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S = 2, 4, 777
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 82)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    o0, l0 = torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    o1, l1 = torch.empty_like(q), torch.empty_like(l0)
    st = torch.cuda.current_stream().cuda_stream
    dt = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    assert fa.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o0.data_ptr(), l0.data_ptr(),
                         B, H, H, S, D, causal, D ** -0.5, dt, st) == fa.FA_OK
    assert fa.fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(),
                             l1.data_ptr(), B, H, H, S, D, causal, 0.0, 99, D ** -0.5, dt,
                             st) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0, l1)


# 1 / (1 - p) is a power of two for these p, so the read-back is exact
@pytest.mark.parametrize("D,dtype,p", [(64, "f16", 0.5), (128, "bf16", 0.5), (128, "bf16", 0.75),
                                       (64, "f16", 0.875), (256, "bf16", 0.5)])
def test_mask_read_back_bit_exact(D, dtype, p):
    """Q = 0 makes every visible probability 1/S; a V whose key j carries a 1
    in column j - c*D only (block c) turns O(1 - p) S into the keep bits of
    keys c*D .. c*D + D - 1, exact in the 16-bit output.  All blocks of keys
    are read, one call each, and compared with the oracle's mask."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S = 2, 3, 4 * D
    seed = 0xDEADBEEF_00C0FFEE
    q = torch.zeros((B, S, H, D), dtype=torch.float16 if dtype == "f16" else torch.bfloat16,
                    device="cuda")
    k = fa_inputs.to_torch(fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 83)[1], dtype).cuda()
    keep = np.empty((B, H, S, S), dtype=bool)
    for c in range(S // D):
        v = torch.zeros_like(q)
        j = torch.arange(c * D, (c + 1) * D, device="cuda")
        v[:, j, :, j - c * D] = 1.0
        o, _ = fa.attention_forward(q, k, v, scale=1.0, dropout_p=p, seed=seed)
        torch.cuda.synchronize()
        bits = (o.double() * ((1.0 - p) * S)).cpu().numpy()   # [B, S, H, D]
        assert np.array_equal(bits, np.round(bits)), "read-back is not integral"
        assert set(np.unique(bits)) <= {0.0, 1.0}
        keep[:, :, :, c * D:(c + 1) * D] = bits.transpose(0, 2, 1, 3) == 1.0
    ref = dropout_keep(B, H, S, p, seed)
    assert np.array_equal(keep, ref), f"{np.count_nonzero(keep != ref)} keep bits differ"
    frac = keep.mean()
    assert abs(frac - (1.0 - p)) < 0.02


def test_dropout_full_size_sampled_rows():
    """The b2h16d128 shape (B=2, H=16, S=8192, D=128 bf16, causal) with
    p = 0.1: a sample of rows of four heads against the oracle, computed for
    those rows only."""
    import torch
    import attention_forward_fwd_gb300 as fa
    from oracle.attention import decode
    from oracle.dropout import dropout_draws, dropout_threshold
    w = fa_inputs.WORKLOADS["b2h16d128"]
    p, seed = 0.1, 2024
    qb, kb, vb = fa_inputs.make_qkv_for(w)
    q, k, v = (fa_inputs.to_torch(x, w.dtype).cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=w.scale, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    O, L = o.double().cpu().numpy(), lse.double().cpu().numpy()
    rng = np.random.default_rng(5)
    thr = np.uint64(dropout_threshold(p))
    for b, h in ((0, 0), (0, 15), (1, 7), (1, 9)):
        rows = np.sort(rng.choice(w.S, 24, replace=False))
        qh = decode(qb[b, rows, h, :], w.dtype)
        kh, vh = decode(kb[b, :, h, :], w.dtype), decode(vb[b, :, h, :], w.dtype)
        z = w.scale * (qh @ kh.T)
        z[np.arange(w.S)[None, :] > rows[:, None]] = -np.inf
        m = z.max(axis=1)
        e = np.exp(z - m[:, None])
        l = e.sum(axis=1)
        keep = dropout_draws(b, h, rows, w.S // 8, seed) >= thr
        Oref = (e * keep / l[:, None]) @ vh / (1.0 - p)
        Lref = m + np.log(l)
        A = (e * keep / l[:, None]) @ np.abs(vh) / (1.0 - p)
        _assert_dropout_close(O[b, rows, h, :], L[b, h, rows], Oref, Lref, A, w.dtype,
                              f"b={b} h={h}")


def test_bad_probability_is_rejected():
    import torch
    import attention_forward_fwd_gb300 as fa
    q = torch.zeros((1, 128, 1, 64), dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    st = torch.cuda.current_stream().cuda_stream
    for bad in (-0.1, 1.0, 1.5, float("nan")):
        assert fa.fa_fwd_dropout(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None,
                                 1, 1, 1, 128, 64, 0, bad, 0, 0.125, fa.FA_F16,
                                 st) == fa.FA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        fa.attention_forward(q, q, q, dropout_p=1.0)
