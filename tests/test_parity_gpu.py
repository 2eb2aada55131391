"""GPU parity: the sm_103a kernel (through the C-ABI) against the fp64 oracle.

Tolerances: |O_gpu - O_ref| <= 2e-3 (fp16) / 8e-3 (bf16) plus half an ulp of
the 16-bit type O is stored in (at O_ref: the final rounding of O to that
type can by itself move it by up to that much), and
|LSE_gpu - LSE_ref| <= 1e-4 |LSE_ref| + 1e-4, the oracle computing the plain
definition in fp64 from the same 16-bit inputs.
"""
import numpy as np
import pytest

import fa_inputs
from oracle import attention_reference, attention_rows

from gpu_common import assert_bare_tolerance, assert_close, o_tol, run_gpu

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


def _full_case(B, H, S, D, dtype, dist, seed, causal, scale=None, ikh=(), split_kv=False):
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, dist, seed, identical_key_head=ikh)
    scale = scale if scale is not None else D ** -0.5
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale, split_kv=split_kv)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale)
    assert_close(O, L, Oref, Lref, dtype,
                 f"B{B} H{H} S{S} D{D} {dtype} causal={causal} split={split_kv}")
    return O, L, Oref, Lref


def _splits(B, H, S, D, causal):
    import attention_forward_fwd_gb300 as fa
    return fa.fa_splitkv_launches(B, H, S, D, causal) == 2


# ------------------------------------------------------------ small / ragged
@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 2, 17, 64, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 640])
def test_ragged_lengths_f16_d64(S, causal, split_kv):
    _full_case(2, 3, S, 64, "f16", "normal", 10 + S, causal, split_kv=split_kv)


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 100, 128, 300, 513])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (128, "f16"), (64, "bf16")])
def test_ragged_lengths_other_types(S, D, dtype, causal, split_kv):
    _full_case(1, 2, S, D, dtype, "normal", 20 + S, causal, split_kv=split_kv)


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
def test_peaky_logits(causal, split_kv):
    """Q, K scaled by 4: max moves by many units across tiles (lazy rescale)."""
    _full_case(1, 4, 700, 64, "f16", "stress", 5, causal, split_kv=split_kv)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (128, "f16")])
def test_peaky_logits_row_split(D, dtype, causal):
    """Peaky scores at D = 128 (two threads per row), several work items per
    CTA: the row sum often rules out the current reference max."""
    _full_case(2, 100, 700, D, dtype, "stress", 6, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (128, "f16")])
def test_rising_scores_move_the_reference(D, dtype, causal):
    """Constant queries and keys that grow along the sequence: every key tile
    lies a little above the previous one (about 2 log2 units per tile), so
    each tile raises the row max by less than the lazy-rescale threshold
    while its row sum exceeds 2^8 against the previous reference."""
    B, H, S = 1, 3, 1024
    rng = np.random.default_rng(12)
    q = np.full((B, S, H, D), 0.5, dtype=np.float32)
    ramp = (2.0 * np.arange(S) / S).astype(np.float32)
    k = np.broadcast_to(ramp[None, :, None, None], (B, S, H, D))
    v = rng.uniform(-1, 1, size=(B, S, H, D)).astype(np.float32)
    qb, kb, vb = (fa_inputs.f32_to_bits(x, dtype) for x in (q, k, v))
    scale = D ** -0.5
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale)
    assert_close(O, L, Oref, Lref, dtype, f"rising D{D} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,D,dtype", [(700, 64, "f16"), (1999, 64, "f16"), (2048, 128, "bf16"),
                                       (3000, 128, "f16"), (4096, 64, "bf16")])
def test_split_kv_path_is_taken_and_exact(S, D, dtype, causal):
    """Shapes with one head: the keys are split over CTAs and the partial
    results merged; the result matches the oracle like the unsplit path."""
    assert _splits(1, 1, S, D, causal)
    _full_case(1, 1, S, D, dtype, "stress", 30 + S, causal, split_kv=True)


@pytest.mark.parametrize("B,H,S,D,dtype,dist", [(1, 40, 1000, 64, "f16", "normal"),
                                                  (1, 40, 900, 128, "bf16", "stress"),
                                                  (3, 8, 1999, 64, "f16", "stress")])
def test_multiwave_split_is_taken_and_exact(B, H, S, D, dtype, dist):
    """One to two waves of query blocks with a ragged last one: some blocks
    are split over CTAs (the plan the host simulation picks), the rest run
    whole in the same launch, and the merge leaves the unsplit blocks alone;
    every element matches the oracle."""
    import torch
    import attention_forward_fwd_gb300 as fa
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits, items = fa.fa_split_plan(B, H, S, D, False, sms)
    assert max(splits) > 1 and min(splits) == 1 and B * H * items > sms
    assert _splits(B, H, S, D, False)
    _full_case(B, H, S, D, dtype, dist, 40 + S, False, split_kv=True)


@pytest.mark.parametrize("S,D,dtype,causal,dist", [(1000, 256, "bf16", False, "normal"),
                                                    (1000, 256, "f16", True, "stress"),
                                                    (2500, 192, "bf16", True, "normal"),
                                                    (4096, 256, "bf16", True, "normal"),
                                                    (300, 136, "f16", False, "normal")])
def test_wide_split_is_taken_and_exact(S, D, dtype, causal, dist):
    """D > 128 with two heads: every query tile's keys are divided over
    several CTAs of the wide kernel (causal: the later chunks of the early
    tiles see no key and are skipped by the merge), and every element
    matches the oracle."""
    assert _splits(1, 2, S, D, causal)
    _full_case(1, 2, S, D, dtype, dist, 50 + S + D, causal, split_kv=True)


def test_split_kv_workspace_checks():
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S, D = 1, 1, 2048, 64
    need = fa.fa_splitkv_workspace_size(B, H, S, D, False)
    assert need > 0
    q = torch.zeros(B, S, H, D, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None, B, H, S, D, 0, 0.125,
            fa.FA_F16)
    assert fa.fa_fwd_splitkv(*args, None, need, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr() + 4, need, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, None) == fa.FA_OK
    torch.cuda.synchronize()
    # a shape that fills the GPU needs no workspace and takes one launch
    assert fa.fa_splitkv_workspace_size(4, 16, 4096, 64, True) == 0
    assert fa.fa_splitkv_launches(4, 16, 4096, 64, True) == 1


@pytest.mark.parametrize("B,H,S,D,dtype,causal", [
    (2, 80, 600, 128, "bf16", True),    # ragged last block: its second query tile is empty
    (2, 80, 600, 128, "bf16", False),
    (2, 80, 600, 64, "f16", True),
    (2, 100, 300, 64, "f16", False),
    (4, 40, 512, 64, "f16", True),
    (2, 40, 1000, 128, "f16", True),
])
def test_several_work_items_per_cta(B, H, S, D, dtype, causal):
    """More query blocks than SMs: each CTA runs several items in turn, so
    barrier phases, the K/V ring, the Q buffer and the O staging carry over
    from one item to the next (including two ragged blocks in a row)."""
    import attention_forward_fwd_gb300 as fa
    import torch
    items = B * H * ((S + 255) // 256)
    assert items > torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.fa_splitkv_launches(B, H, S, D, causal) == 1
    _full_case(B, H, S, D, dtype, "normal", 40 + S, causal)


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,H_kv,S,D,dtype", [
    (2, 8, 2, 300, 64, "f16"),     # GQA, ragged
    (1, 8, 1, 513, 64, "bf16"),    # MQA
    (2, 16, 4, 640, 128, "bf16"),
    (1, 6, 3, 257, 128, "f16"),
    (3, 40, 8, 512, 64, "f16"),    # several work items per CTA
])
def test_grouped_kv_heads(B, H, H_kv, S, D, dtype, causal, split_kv):
    """K/V with H_kv heads shared by groups of H / H_kv query heads, every
    element against the oracle (one CTA per block and the key split)."""
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 50 + S + H_kv, h_kv=H_kv)
    scale = D ** -0.5
    O, L = run_gpu(qb, kb, vb, dtype, causal, scale, split_kv=split_kv)
    Oref, Lref = attention_reference(qb, kb, vb, dtype, causal, scale)
    assert_close(O, L, Oref, Lref, dtype, f"B{B} H{H}/{H_kv} S{S} D{D} {dtype} causal={causal}")


def test_grouped_kv_heads_split_path_is_taken():
    """One query head group on a long sequence: the keys are split and merged."""
    import attention_forward_fwd_gb300 as fa
    assert fa.fa_splitkv_launches(1, 2, 3000, 64, True) == 2
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 3000, 64, "f16", "stress", 77, h_kv=1)
    O, L = run_gpu(qb, kb, vb, "f16", True, 0.125, split_kv=True)
    Oref, Lref = attention_reference(qb, kb, vb, "f16", True, 0.125)
    assert_close(O, L, Oref, Lref, "f16", "MQA split")


def test_many_heads_and_batches_layout():
    """[B, S, H, D] with H > 1 and B > 1: heads and batches land in place."""
    _full_case(3, 5, 200, 64, "f16", "normal", 6, False)
    _full_case(3, 5, 200, 128, "bf16", "normal", 7, True)


# ------------------------------------------------------------- the workloads
def test_workload_s256():
    w = fa_inputs.WORKLOADS["s256"]
    qb, kb, vb = fa_inputs.make_qkv_for(w)
    for causal in w.modes:
        O, L = run_gpu(qb, kb, vb, w.dtype, causal, w.scale)
        Oref, Lref = attention_reference(qb, kb, vb, w.dtype, causal, w.scale)
        assert_close(O, L, Oref, Lref, w.dtype, "s256")
        assert_bare_tolerance(O, Oref, w.dtype, "s256")


@pytest.mark.parametrize("split_kv", [False, True], ids=["one-cta-per-block", "split-kv"])
@pytest.mark.parametrize("causal", [False, True])
def test_workload_s4096(causal, split_kv):
    w = fa_inputs.WORKLOADS["s4096"]
    qb, kb, vb = fa_inputs.make_qkv_for(w)
    O, L = run_gpu(qb, kb, vb, w.dtype, causal, w.scale, split_kv=split_kv)
    Oref, Lref = attention_reference(qb, kb, vb, w.dtype, causal, w.scale)
    assert_close(O, L, Oref, Lref, w.dtype, f"s4096 causal={causal} split={split_kv}")
    assert_bare_tolerance(O, Oref, w.dtype, "s4096")


@pytest.mark.parametrize("causal", [True, False])
def test_workload_stress_full(causal):
    """B=3,H=8,S=1999 peaky logits, every element against the oracle; the
    identical-key head equals the (prefix) mean of V."""
    w = fa_inputs.WORKLOADS["stress"]
    qb, kb, vb = fa_inputs.make_qkv_for(w)
    O, L = run_gpu(qb, kb, vb, w.dtype, causal, w.scale)
    Oref, Lref = attention_reference(qb, kb, vb, w.dtype, causal, w.scale)
    assert_close(O, L, Oref, Lref, w.dtype, f"stress causal={causal}")
    assert_bare_tolerance(O, Oref, w.dtype, "stress")
    b, h = w.identical_key_head
    v = Oref[b, :, h, :]
    assert np.all(np.abs(O[b, :, h, :] - v) <= o_tol(v, "f16"))


def _sampled_rows(S, rng, n=24):
    fixed = [0, 1, 127, 128, 129, 255, 256, 257, S // 2, S - 129, S - 128, S - 2, S - 1]
    rows = set(r for r in fixed if 0 <= r < S)
    rows.update(rng.integers(0, S, size=n - len(rows)).tolist())
    return sorted(rows)


@pytest.mark.parametrize("name,causal", [("b4h16", True), ("b2h16d128", True),
                                         ("b2h16d128", False), ("b4h32kv8d128", True)])
def test_workload_full_size_sampled(name, causal):
    """Full-size workloads in the launch configuration the bench times,
    against the oracle row by row: the first and the last 256-row query
    block of every head (the lightest and heaviest work items when causal,
    the ragged end), and sampled rows of six heads."""
    w = fa_inputs.WORKLOADS[name]
    qb, kb, vb = fa_inputs.make_qkv_for(w)
    O, L = run_gpu(qb, kb, vb, w.dtype, causal, w.scale)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    edge = sorted(set(range(min(256, w.S))) | set(range(max(0, w.S - 256), w.S)))
    for b in range(w.B):
        for h in range(w.H):
            Oref, Lref = attention_rows(qb, kb, vb, w.dtype, causal, w.scale, b, h, edge)
            what = f"{name} causal={causal} b{b} h{h} first/last block"
            assert_close(O[b, edge, h, :], L[b, h, edge], Oref, Lref, w.dtype, what)
            assert_bare_tolerance(O[b, edge, h, :], Oref, w.dtype, what)
    rng = np.random.default_rng(123)
    heads = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H)))
                                            for _ in range(4)]
    for b, h in heads:
        rows = _sampled_rows(w.S, rng)
        Oref, Lref = attention_rows(qb, kb, vb, w.dtype, causal, w.scale, b, h, rows)
        assert_close(O[b, rows, h, :], L[b, h, rows], Oref, Lref, w.dtype, f"{name} b{b} h{h}")


# ------------------------------------------------------------ API behaviour
def test_no_lse_pointer():
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 300, 64, "f16", "normal", 8)
    O, L = run_gpu(qb, kb, vb, "f16", True, 0.125, with_lse=False)
    assert L is None
    Oref, _ = attention_reference(qb, kb, vb, "f16", True, 0.125)
    assert np.all(np.abs(O - Oref) <= o_tol(Oref, "f16"))


def test_side_stream_and_repeatability():
    """Bit-identical results over repeated calls on a non-default stream."""
    import torch
    import attention_forward_fwd_gb300 as fa
    qb, kb, vb = fa_inputs.make_qkv(2, 4, 1000, 64, "f16", "stress", 9)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(10):
            o, lse = fa.attention_forward(q, k, v, causal=True, scale=0.125)
            outs.append((o.clone(), lse.clone()))
    s.synchronize()
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_output_written_only_inside_the_tensor():
    """Rows past S must not be written: surround O with guard bands."""
    import torch
    import attention_forward_fwd_gb300 as fa
    B, H, S, D = 1, 2, 300, 64
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "f16", "normal", 11)
    q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
    n = B * S * H * D
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=torch.float16, device="cuda")
    o = buf[guard:guard + n].view(B, S, H, D)
    lbuf = torch.full((B * H * S + 2 * 64,), 3.0, dtype=torch.float32, device="cuda")
    lse = lbuf[64:64 + B * H * S].view(B, H, S)
    fa.attention_forward(q, k, v, causal=False, scale=0.125, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)
    assert torch.all(lbuf[:64] == 3.0) and torch.all(lbuf[64 + B * H * S:] == 3.0)
    Oref, Lref = attention_reference(qb, kb, vb, "f16", False, 0.125)
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, "f16")


def test_stream_argument_with_a_split_call():
    """A torch stream object passed as ``stream=`` (not made current): the
    split path's workspace is allocated for that stream, the call runs there,
    and the result matches the oracle; a second shape that needs a larger
    workspace (about 1.1 MB, then 9.7 MB on 152 SMs) replaces the cached
    buffer of that stream."""
    import torch
    import attention_forward_fwd_gb300 as fa
    s = torch.cuda.Stream()
    key = (str(torch.device("cuda", torch.cuda.current_device())), int(s.cuda_stream))
    fa._WORKSPACES.pop(key, None)   # stream handles are recycled by torch's pool
    sizes = []
    for S, seed in ((1024, 21), (3000, 22)):
        need = fa.fa_splitkv_workspace_size(1, 1, S, 64, False)
        assert need > 0
        qb, kb, vb = fa_inputs.make_qkv(1, 1, S, 64, "f16", "normal", seed)
        q, k, v = (fa_inputs.to_torch(x, "f16").cuda() for x in (qb, kb, vb))
        torch.cuda.synchronize()
        o, lse = fa.attention_forward(q, k, v, causal=False, scale=0.125, stream=s)
        s.synchronize()
        assert fa._WORKSPACES[key].numel() >= need
        sizes.append(fa._WORKSPACES[key].numel())
        Oref, Lref = attention_reference(qb, kb, vb, "f16", False, 0.125)
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, "f16",
                     f"S{S} on a stream object")
    if fa.fa_splitkv_workspace_size(1, 1, 3000, 64, False) > sizes[0]:
        assert sizes[1] > sizes[0]
