"""The debug build (FA_DEBUG = 1) against the release build.

libfa_gb300_debug.so compiles the same sources with device-side invariant
checks: every work item's key-tile range lies inside its sequence and its
split fields in range, tensor memory is allocated from column 0, the
producer and the MMA warps saw the same ring of K / V tiles and the softmax
read every S the MMA warps issued, every stored row's sum is positive, and
every merged query block has between 1 and max_splits splits.  A failed
check records FA_ERR_DEVICE_CHECK in that library's own status word; it
never traps.  Here every entry point family runs through both libraries on
the same device inputs: the outputs must be bit for bit the same (the checks
do not touch the arithmetic) and no check may fire.
"""
import ctypes

import numpy as np
import pytest

import fa_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    import torch
    import attention_forward_fwd_gb300 as fa
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    fa.build()
    rel, dbg = fa.library(), fa.debug_library()
    rel.fa_device_status(1)
    dbg.fa_device_status(1)
    yield rel, dbg
    assert dbg.fa_device_status(1) == 0, "a device-side check failed in the debug build"


def _dev(x, dtype):
    return fa_inputs.to_torch(x, dtype).cuda()


def _both(libs, run):
    """run(lib) -> (O, LSE) tensors; returns both libraries' results."""
    import torch
    outs = [run(lib) for lib in libs]
    torch.cuda.synchronize()
    return outs


def _same(outs, what):
    import torch
    (o1, l1), (o2, l2) = outs
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), f"{what}: O differs"
    assert torch.equal(l1, l2), f"{what}: LSE differs"


SPLITKV = [
    # (B, H, H_kv, S, D, dtype, causal, dist)
    (2, 3, 3, 1000, 64, "f16", True, "normal"),      # one wave: split
    (1, 1, 1, 4096, 64, "f16", False, "normal"),     # one wave: split
    (3, 8, 8, 1999, 64, "f16", False, "stress"),     # ragged waves: multi-wave split plan
    (4, 16, 16, 1024, 64, "f16", True, "normal"),    # several items per CTA
    (2, 4, 2, 777, 128, "bf16", False, "normal"),    # grouped K/V heads
    (2, 16, 16, 2048, 128, "bf16", True, "normal"),  # several items per CTA
    (1, 2, 1, 1500, 256, "bf16", True, "normal"),    # the wide kernel
    (1, 3, 3, 900, 176, "f16", False, "normal"),     # the wide kernel at width 192
]


@pytest.mark.parametrize("B,H,H_kv,S,D,dtype,causal,dist", SPLITKV)
def test_splitkv_entry(libs, B, H, H_kv, S, D, dtype, causal, dist):
    import torch
    import attention_forward_fwd_gb300 as fa
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, dist, 900 + S + D, h_kv=H_kv)
    q, k, v = (_dev(x, dtype) for x in (qb, kb, vb))
    code = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    n = ctypes.c_size_t(0)
    assert libs[0].fa_splitkv_workspace_size(B, H, S, D, int(causal), ctypes.byref(n)) == 0
    ws = torch.empty(max(int(n.value), 16), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    def run(lib):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
        rc = lib.fa_fwd_gqa_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    B, H, H_kv, S, D, int(causal), D ** -0.5, code, ws.data_ptr(), ws.numel(), st)
        assert rc == 0, rc
        return o, lse
    _same(_both(libs, run), f"splitkv B{B} H{H}/{H_kv} S{S} D{D} causal={causal}")


@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16")])
def test_varlen_local_dropout_entries(libs, D, dtype):
    import torch
    import attention_forward_fwd_gb300 as fa
    code = fa.FA_F16 if dtype == "f16" else fa.FA_BF16
    st = torch.cuda.current_stream().cuda_stream
    scale = D ** -0.5

    # packed variable-length batch
    lens = fa_inputs.varlen_lengths(9, 1, 900, 31 + D)
    qb, kb, vb, cu = fa_inputs.make_varlen(lens, 4, D, dtype, "normal", 32 + D, h_kv=2)
    q, k, v = (_dev(x, dtype) for x in (qb, kb, vb))
    cu_d = torch.from_numpy(cu).cuda()
    total, smax = int(cu[-1]), int(np.max(lens))

    def run_varlen(lib):
        o = torch.empty_like(q)
        lse = torch.empty((4, total), dtype=torch.float32, device="cuda")
        rc = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               cu_d.data_ptr(), len(lens), smax, total, 4, 2, D, 1, scale, code, st)
        assert rc == 0, rc
        return o, lse
    _same(_both(libs, run_varlen), f"varlen D{D}")

    # sliding window and dropout on one batched shape
    B, H, S = 2, 4, 1300
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dtype, "normal", 33 + D)
    q, k, v = (_dev(x, dtype) for x in (qb, kb, vb))

    def run_local(lib):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
        rc = lib.fa_fwd_local(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              B, H, H, S, D, 1, 300, -1, scale, code, st)
        assert rc == 0, rc
        return o, lse
    _same(_both(libs, run_local), f"local D{D}")

    def run_dropout(lib):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
        rc = lib.fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, H, S, D, 0, 0.1, 1234, scale, code, st)
        assert rc == 0, rc
        return o, lse
    _same(_both(libs, run_dropout), f"dropout D{D}")
