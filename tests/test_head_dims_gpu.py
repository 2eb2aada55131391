"""GPU parity for head dimensions other than 64 and 128 against the fp64
oracle.  A head dimension D (a multiple of 8 up to 256) runs on the D = 64,
D = 128, D = 192 or D = 256 kernel, whose tensor maps cover only the D
columns: the copies read the others as zeros and the O stores leave them out.  Every path that stores
O is covered: the TMA store, the merge of split keys and the row-by-row
stores of a packed sequence's last tile, with guard bands around O.
Tolerances as in test_parity_gpu.py."""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference, attention_reference_varlen, attention_rows
from oracle.dropout import attention_reference_dropout

from gpu_common import TOL_O, assert_close, half_ulp, lse_tol, run_gpu

pytestmark = pytest.mark.gpu

DIMS = [8, 16, 32, 40, 48, 56, 72, 80, 96, 112, 120]


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


def _dtype(D):
    return "bf16" if D % 16 else "f16"


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", DIMS)
def test_head_dims(D, causal, split_kv):
    import attention_forward_fwd_gb300 as fa
    B, H, S = 1, 2, 700
    dtype = _dtype(D)
    if split_kv:
        assert fa.fa_splitkv_workspace_size(B, H, S, D, causal) > 0
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 100 + D)
    O, L = run_gpu(qb, kb, vb, dtype, causal, D ** -0.5, split_kv=split_kv)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, D ** -0.5)
    assert_close(O, L, Oref, Lref, dtype, f"D{D} causal={causal} split={split_kv}")


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("D", [24, 96, 176, 232])
def test_output_stays_inside_the_tensor(D, split_kv):
    """O surrounded by guard bands: no column past D and no row past S is
    written (rows are D elements apart, not the kernel's width)."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S = 1, 3, 555
    dtype = _dtype(D)
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "stress", 110 + D)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    n = B * S * H * D
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=q.dtype, device="cuda")
    o = buf[guard:guard + n].view(B, S, H, D)
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=D ** -0.5, out=o, split_kv=split_kv)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, True, D ** -0.5)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                 f"guarded D{D}")


@pytest.mark.parametrize("D", [32, 96, 192, 256])
def test_packed_batch_row_stores(D):
    """Packed sequences whose last tiles are stored row by row, with the
    next sequence's rows right after them (D > 128: the wide kernel, which
    stores every row itself)."""
    import torch
    import attention_forward_fwd_gb300 as fa
    dtype = _dtype(D)
    lens = [1, 130, 257, 0, 300, 77]
    qb, kb, vb, cu = fa_inputs.make_varlen(lens, 4, D, dtype, "normal", 120 + D, h_kv=2)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = fa.attention_forward_varlen(q, k, v, cu_t, max(lens), causal=True, scale=D ** -0.5)
    torch.cuda.synchronize()
    Oref, Lref = attention_reference_varlen(qb, kb, vb, cu, dtype, True, D ** -0.5)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                 f"packed D{D}")


def test_grouped_heads_window_and_dropout_at_other_dims():
    import torch
    import attention_forward_fwd_gb300 as fa
    # grouped K/V heads (8 query heads over 2), D = 40
    qb, kb, vb = fa_inputs.make_qkv(2, 8, 400, 40, "bf16", "normal", 131, h_kv=2)
    O, L = run_gpu(qb, kb, vb, "bf16", True, 40 ** -0.5)
    Oref, Lref = attention_reference(qb, kb, vb, "bf16", True, 40 ** -0.5)
    assert_close(O, L, Oref, Lref, "bf16", "GQA D40")
    # sliding window, D = 96
    qb, kb, vb = fa_inputs.make_qkv(1, 4, 900, 96, "f16", "normal", 132)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=96 ** -0.5, window=(200, -1))
    torch.cuda.synchronize()
    Oref, Lref = attention_reference(qb, kb, vb, "f16", True, 96 ** -0.5, window=(200, -1))
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, "f16",
                 "window D96")
    # dropout, D = 48
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 333, 48, "f16", "normal", 133)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=False, scale=48 ** -0.5, dropout_p=0.25, seed=5)
    torch.cuda.synchronize()
    Oref, Lref = attention_reference_dropout(qb, kb, vb, "f16", False, 48 ** -0.5, 0.25, 5)
    # the dropout tests' bound: the forward's tolerance times 1 / (1 - p)
    d = np.abs(o.double().cpu().numpy() - Oref)
    assert np.all(d <= TOL_O["f16"] / 0.75 + half_ulp(Oref, "f16")), d.max()
    assert np.all(np.abs(lse.double().cpu().numpy() - Lref) <= lse_tol(Lref))


def test_head_dim_96_full_size_sampled_rows():
    """B2 H16 S8192 D96 bf16, causal (the b2h16d128 shape with D = 96): sampled
    rows of a few heads against the oracle, computed for those rows only."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S, D = 2, 16, 8192, 96
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "bf16", "normal", 134)
    q, k, v = (fa_inputs.to_torch(x, "bf16").cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=D ** -0.5)
    torch.cuda.synchronize()
    O, L = o.double().cpu().numpy(), lse.double().cpu().numpy()
    rng = np.random.default_rng(9)
    for b, h in ((0, 0), (1, 15), (0, 9)):
        rows = np.sort(np.concatenate([rng.choice(S, 20, replace=False), [0, S - 1]]))
        Oref, Lref = attention_rows(qb, kb, vb, "bf16", True, D ** -0.5, b, h, rows)
        assert_close(O[b, rows, h, :], L[b, h, rows], Oref, Lref, "bf16", f"D96 b={b} h={h}")


# ------------------------------------------------- D > 128: the wide kernel
WIDE = [136, 160, 192, 200, 248, 256]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", WIDE)
def test_wide_head_dims(D, causal):
    """Several query tiles, a ragged last tile, grouped K/V heads."""
    B, H, H_kv, S = 2, 4, 2, 333
    dtype = "bf16" if D % 16 else "f16"
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 140 + D, h_kv=H_kv)
    O, L = run_gpu(qb, kb, vb, dtype, causal, D ** -0.5)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, D ** -0.5)
    assert_close(O, L, Oref, Lref, dtype, f"D{D} causal={causal}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_wide_peaky_scores_and_guard_bands(dtype):
    """Peaky scores (the reference max moves, O is rescaled) and guard bands
    around O; three heads leave most SMs idle, so the split entry point
    divides the wide kernel's key tiles and the merge kernel writes O."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S, D = 1, 3, 700, 256
    assert fa.fa_splitkv_workspace_size(B, H, S, D, True) > 0
    assert fa.fa_splitkv_launches(B, H, S, D, True) == 2
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "stress", 150)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    n = B * S * H * D
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=q.dtype, device="cuda")
    o = buf[guard:guard + n].view(B, S, H, D)
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=D ** -0.5, out=o)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, True, D ** -0.5)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype, "stress D256")


@pytest.mark.parametrize("D,window,causal,H_kv", [(256, (300, -1), True, 3), (192, (200, 150), False, 1),
                                                   (256, (0, 0), False, 3), (136, (129, 40), True, 1)])
def test_wide_window(D, window, causal, H_kv):
    """Sliding windows on the wide kernel (D > 128): key-tile ranges per query
    tile, rows whose first tiles lie wholly outside their window, grouped
    K/V heads; every element against the oracle."""
    import attention_forward_fwd_gb300 as fa
    dtype = "bf16"
    B, H, S = 2, 3, 1100
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 160 + D + window[0], h_kv=H_kv)
    q, k, v = (fa_inputs.to_torch(x, dtype).cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=D ** -0.5, window=window)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, D ** -0.5, window=window)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, dtype,
                 f"window {window} D{D} causal={causal}")


@pytest.mark.parametrize("D", [192, 256])
def test_wide_full_size_sampled_rows(D):
    """B2 H16 S8192 bf16 at D = 192 and 256, causal: sampled rows of a few heads."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S = 2, 16, 8192
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "bf16", "normal", 151 + D % 256)
    q, k, v = (fa_inputs.to_torch(x, "bf16").cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=D ** -0.5)
    torch.cuda.synchronize()
    O, L = o.double().cpu().numpy(), lse.double().cpu().numpy()
    rng = np.random.default_rng(10)
    for b, h in ((0, 0), (1, 15), (1, 4)):
        rows = np.sort(np.concatenate([rng.choice(S, 20, replace=False), [0, S - 1]]))
        Oref, Lref = attention_rows(qb, kb, vb, "bf16", True, D ** -0.5, b, h, rows)
        assert_close(O[b, rows, h, :], L[b, h, rows], Oref, Lref, "bf16", f"D{D} b={b} h={h}")


@pytest.mark.parametrize("S", [1, 2, 127, 129, 255, 257, 383])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [192, 256])
def test_wide_edge_lengths(D, S, causal):
    """One key, tile boundaries and lengths that are not multiples of 8."""
    dtype = "f16"
    qb, kb, vb = fa_inputs.make_qkv(1, 2, S, D, dtype, "stress", 160 + S + D)
    O, L = run_gpu(qb, kb, vb, dtype, causal, D ** -0.5)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, D ** -0.5)
    assert_close(O, L, Oref, Lref, dtype, f"D{D} S{S} causal={causal}")


def test_wide_many_heads_one_wave_and_more():
    """More CTAs than SMs (B4 H40 S300 -> 480 CTAs), grouped K/V heads."""
    B, H, H_kv, S, D = 4, 40, 8, 300, 192
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "bf16", "normal", 170, h_kv=H_kv)
    O, L = run_gpu(qb, kb, vb, "bf16", True, D ** -0.5)
    Oref, Lref = attention_reference(qb, kb, vb, "bf16", True, D ** -0.5)
    assert_close(O, L, Oref, Lref, "bf16", "D192 many heads")


@pytest.mark.parametrize("H,H_kv,causal", [(6, 2, True), (5, 1, False)])
def test_wide_partial_last_head_group(H, H_kv, causal):
    """The wide kernel numbers its CTAs by groups of heads whose K and V fit
    in 32 MB (causal) or 16 MB (non-causal) together: at S = 8192, D = 256
    that is 4 or 2 heads, so 6 causal query heads form groups of 4 and 2, and
    5 non-causal ones groups of 2, 2 and 1 (grouped K/V heads in both).
    Sampled rows of every head."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, S, D = 1, 8192, 256
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "bf16", "normal", 171 + H, h_kv=H_kv)
    q, k, v = (fa_inputs.to_torch(x, "bf16").cuda() for x in (qb, kb, vb))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=D ** -0.5)
    torch.cuda.synchronize()
    O, L = o.double().cpu().numpy(), lse.double().cpu().numpy()
    rng = np.random.default_rng(11)
    for h in range(H):
        rows = np.sort(np.concatenate([rng.choice(S, 12, replace=False), [0, S - 1]]))
        Oref, Lref = attention_rows(qb, kb, vb, "bf16", causal, D ** -0.5, 0, h, rows)
        assert_close(O[0, rows, h, :], L[0, h, rows], Oref, Lref, "bf16", f"D256 h={h}")


@pytest.mark.parametrize("D,width", [(136, 192), (176, 192), (192, 192), (200, 256), (256, 256)])
def test_wide_split_workspace_has_the_kernel_width(D, width):
    """D = 136 .. 192 run on the 192-column kernel, 200 .. 256 on the
    256-column one; a split call's partials have the kernel's width (fp32 o~
    of 128 x width plus m and l per slot), so the workspace scales with it."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S = 1, 2, 1000
    n = fa.fa_splitkv_workspace_size(B, H, S, D, False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits, _ = fa.fa_split_plan(B, H, S, D, False, sms)
    assert max(splits) > 1
    slots = B * H * ((S + 127) // 128) * max(splits)
    assert n == slots * (128 * width + 2 * 128) * 4
