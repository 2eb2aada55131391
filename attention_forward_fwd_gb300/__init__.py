"""FlashAttention-2 forward pass on one GB300 (sm_103a).

Thin Python binding over the C-ABI of ``libfa_gb300.so`` (declared in
``include/fa_gb300.h``).  This module only marshals arguments: every step of
the computation runs in the library's CUDA kernel, on the caller's stream.
There is no CPU or PyTorch fallback; if the library is missing the call
raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH, build  # noqa: F401

__all__ = ["fa_fwd", "fa_fwd_f16", "fa_fwd_bf16", "fa_status_string",
           "fa_device_status", "fa_last_device_status", "attention_forward",
           "fa_fwd_splitkv", "fa_splitkv_workspace_size", "fa_splitkv_launches", "fa_split_plan",
           "fa_fwd_gqa", "fa_fwd_gqa_splitkv", "fa_fwd_varlen", "attention_forward_varlen",
           "fa_fwd_local", "fa_fwd_dropout",
           "FaError", "library", "EXPORTED_SYMBOLS", "FA_F16", "FA_BF16"]

(FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT,
 FA_ERR_BAD_SEQLENS, FA_ERR_DEVICE_CHECK) = range(7)
FA_F16, FA_BF16 = 0, 1

EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_f16", "fa_fwd_bf16", "fa_status_string",
                    "fa_device_status", "fa_last_device_status", "fa_splitkv_workspace_size",
                    "fa_splitkv_launches", "fa_fwd_splitkv", "fa_fwd_gqa", "fa_fwd_gqa_splitkv",
                    "fa_fwd_varlen", "fa_fwd_local", "fa_selftest_timeout", "fa_fwd_dropout",
                    "fa_split_plan")

_LIB = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)} (status {status})")


def library() -> ctypes.CDLL:
    """Load libfa_gb300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "attention_forward_fwd_gb300.build()")
        _LIB = _declare(ctypes.CDLL(LIB_PATH))
    return _LIB


_DEBUG_LIB = None


def debug_library() -> ctypes.CDLL:
    """Build (if needed) and load libfa_gb300_debug.so: the same C-ABI with
    the device-side invariant checks, which report FA_ERR_DEVICE_CHECK
    through its own fa_device_status.  A separate library with a status word
    of its own; for tests."""
    global _DEBUG_LIB
    if _DEBUG_LIB is None:
        _DEBUG_LIB = _declare(ctypes.CDLL(build(debug=True)))
    return _DEBUG_LIB


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Argument and result types of every exported function."""
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = [vp, vp, vp, vp, vp, i, i, i, i, i, f]
    lib.fa_fwd.argtypes = sig + [i, vp]
    lib.fa_fwd_f16.argtypes = sig + [vp]
    lib.fa_fwd_bf16.argtypes = sig + [vp]
    for fn in (lib.fa_fwd, lib.fa_fwd_f16, lib.fa_fwd_bf16):
        fn.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_device_status.argtypes = [i]
    lib.fa_device_status.restype = i
    lib.fa_last_device_status.argtypes = [vp]
    lib.fa_last_device_status.restype = i
    lib.fa_splitkv_workspace_size.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_splitkv_workspace_size.restype = i
    lib.fa_splitkv_launches.argtypes = [i, i, i, i, i]
    lib.fa_splitkv_launches.restype = i
    lib.fa_split_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(i), i, ctypes.POINTER(i)]
    lib.fa_split_plan.restype = i
    lib.fa_fwd_splitkv.argtypes = sig + [i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_splitkv.restype = i
    gsig = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i]   # ..., B, H, H_kv, S, D, causal, scale, dtype
    lib.fa_fwd_gqa.argtypes = gsig + [vp]
    lib.fa_fwd_gqa.restype = i
    lib.fa_fwd_gqa_splitkv.argtypes = gsig + [vp, ctypes.c_size_t, vp]
    lib.fa_fwd_gqa_splitkv.restype = i
    # Q, K, V, O, LSE, cu_seqlens, B, max_seqlen, total, H, H_kv, D, causal, scale, dtype, stream
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.restype = i
    # ..., B, H, H_kv, S, D, causal, window_left, window_right, scale, dtype, stream
    lib.fa_fwd_local.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_local.restype = i
    lib.fa_selftest_timeout.argtypes = [vp, vp, vp, vp, i, i, i, vp]
    # ..., B, H, H_kv, S, D, causal, p_drop, seed, scale, dtype, stream
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_double,
                                   ctypes.c_ulonglong, f, i, vp]
    lib.fa_fwd_dropout.restype = i
    lib.fa_selftest_timeout.restype = i
    return lib


def fa_status_string(status: int) -> str:
    return library().fa_status_string(int(status)).decode()


def fa_device_status(clear: bool = False) -> int:
    return int(library().fa_device_status(1 if clear else 0))


def fa_last_device_status(stream=None) -> int:
    """The device status word after the work enqueued on `stream` so far
    (a torch stream, a raw handle, or None for the current stream); waits
    for that stream only and does not clear the word."""
    return int(library().fa_last_device_status(_stream_handle(stream)))


def fa_fwd(Q, K, V, O, LSE, B, H, S, D, causal, scale, dtype, stream) -> int:
    """Raw C-ABI call with integer device pointers; returns the status."""
    return int(library().fa_fwd(Q, K, V, O, LSE, int(B), int(H), int(S), int(D),
                                int(bool(causal)), float(scale), int(dtype), stream))


def fa_fwd_f16(Q, K, V, O, LSE, B, H, S, D, causal, scale, stream) -> int:
    return int(library().fa_fwd_f16(Q, K, V, O, LSE, int(B), int(H), int(S), int(D),
                                    int(bool(causal)), float(scale), stream))


def fa_fwd_bf16(Q, K, V, O, LSE, B, H, S, D, causal, scale, stream) -> int:
    return int(library().fa_fwd_bf16(Q, K, V, O, LSE, int(B), int(H), int(S), int(D),
                                     int(bool(causal)), float(scale), stream))


def fa_splitkv_workspace_size(B, H, S, D, causal) -> int:
    """Workspace bytes fa_fwd_splitkv needs on the current device (0: no split)."""
    n = ctypes.c_size_t(0)
    rc = int(library().fa_splitkv_workspace_size(int(B), int(H), int(S), int(D),
                                                 int(bool(causal)), ctypes.byref(n)))
    if rc != FA_OK:
        raise FaError(rc, "fa_splitkv_workspace_size")
    return int(n.value)


def fa_splitkv_launches(B, H, S, D, causal) -> int:
    return int(library().fa_splitkv_launches(int(B), int(H), int(S), int(D), int(bool(causal))))


def fa_split_plan(B, H, S, D, causal, sms):
    """(splits of each 256-row query block, work items per head) of the split
    plan for this shape on a GPU with `sms` SMs (host only, no CUDA call)."""
    nqb = (int(S) + 255) // 256
    arr = (ctypes.c_int * max(nqb, 1))()
    items = ctypes.c_int(0)
    rc = library().fa_split_plan(int(B), int(H), int(S), int(D), int(bool(causal)), int(sms), arr,
                                 nqb, ctypes.byref(items))
    if rc < 1:
        raise FaError(rc, "fa_split_plan")
    return list(arr[:nqb]), items.value


def fa_fwd_splitkv(Q, K, V, O, LSE, B, H, S, D, causal, scale, dtype, workspace,
                   workspace_bytes, stream) -> int:
    """Raw C-ABI call of the split-over-keys entry point; returns the status."""
    return int(library().fa_fwd_splitkv(Q, K, V, O, LSE, int(B), int(H), int(S), int(D),
                                        int(bool(causal)), float(scale), int(dtype),
                                        workspace, int(workspace_bytes), stream))


def fa_fwd_gqa(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype, stream) -> int:
    """Raw C-ABI call with H_kv K/V heads; returns the status."""
    return int(library().fa_fwd_gqa(Q, K, V, O, LSE, int(B), int(H), int(H_kv), int(S), int(D),
                                    int(bool(causal)), float(scale), int(dtype), stream))


def fa_fwd_gqa_splitkv(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype, workspace,
                       workspace_bytes, stream) -> int:
    """Raw C-ABI call with H_kv K/V heads, keys split when SMs would idle."""
    return int(library().fa_fwd_gqa_splitkv(Q, K, V, O, LSE, int(B), int(H), int(H_kv), int(S),
                                            int(D), int(bool(causal)), float(scale), int(dtype),
                                            workspace, int(workspace_bytes), stream))


def fa_fwd_local(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, window_left, window_right, scale,
                 dtype, stream) -> int:
    """Raw C-ABI call with a sliding window (keys i - left .. i + right)."""
    return int(library().fa_fwd_local(Q, K, V, O, LSE, int(B), int(H), int(H_kv), int(S), int(D),
                                      int(bool(causal)), int(window_left), int(window_right),
                                      float(scale), int(dtype), stream))


def fa_fwd_dropout(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, p_drop, seed, scale, dtype,
                   stream) -> int:
    """Raw C-ABI call with attention dropout (probability p_drop, Philox seed)."""
    return int(library().fa_fwd_dropout(Q, K, V, O, LSE, int(B), int(H), int(H_kv), int(S), int(D),
                                        int(bool(causal)), float(p_drop),
                                        int(seed) & 0xFFFFFFFFFFFFFFFF, float(scale), int(dtype),
                                        stream))


def fa_fwd_varlen(Q, K, V, O, LSE, cu_seqlens, B, max_seqlen, total, H, H_kv, D, causal, scale,
                  dtype, stream) -> int:
    """Raw C-ABI call on a packed variable-length batch; returns the status."""
    return int(library().fa_fwd_varlen(Q, K, V, O, LSE, cu_seqlens, int(B), int(max_seqlen),
                                       int(total), int(H), int(H_kv), int(D), int(bool(causal)),
                                       float(scale), int(dtype), stream))


# workspace buffers of the split path, one per (device, stream): calls on one
# stream are ordered, so they may share it
_WORKSPACES = {}


def _workspace(device, stream_handle: int, nbytes: int):
    """The cached workspace of (device, stream), grown to nbytes.  It is
    allocated while the call's own stream is current, so that the caching
    allocator hands a replaced buffer's memory out again only in that
    stream's order, after the kernels that still read it."""
    import torch
    key = (str(device), int(stream_handle))
    buf = _WORKSPACES.get(key)
    if buf is None or buf.numel() < nbytes:
        _WORKSPACES.pop(key, None)
        target = next((st for st in (torch.cuda.current_stream(device),
                                     torch.cuda.default_stream(device))
                       if st.cuda_stream == stream_handle), None)
        if target is None:
            target = torch.cuda.ExternalStream(stream_handle, device=device)
        with torch.cuda.stream(target):
            buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = buf
    return buf


def _stream_handle(stream) -> int:
    """The cudaStream_t of `stream`: None (torch's current stream), a torch
    stream object, or a raw handle."""
    import torch
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _check_devices(device, **tensors):
    """Every tensor given must live on `device` (the kernels take raw pointers
    and would read another GPU's memory through them)."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, q on {device}")


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None,
                      out=None, lse=None, with_lse: bool = True, stream=None,
                      split_kv: bool = True, window=None, dropout_p: float = 0.0,
                      seed: int = 0):
    """O, LSE for torch CUDA tensors q [B, S, H, D] and k, v [B, S, H_kv, D].

    q, k, v must be contiguous fp16 or bf16 tensors on the same CUDA device;
    H_kv must divide H (query head h uses K/V head h // (H / H_kv)); D is a
    multiple of 8 up to 256.
    ``out`` / ``lse`` may be preallocated ([B, S, H, D] same dtype; [B, H, S]
    fp32), on q's device.  Work is enqueued on ``stream`` (a torch stream or
    a raw handle; default: the current stream) and not waited for.  ``split_kv`` lets the library split the keys of each
    query block over several CTAs when the shape leaves SMs idle (the
    workspace is allocated with torch and cached per device and stream).
    ``window = (left, right)`` restricts query i to keys i - left .. i + right
    (-1: no bound on that side); windowed calls are not split.
    ``dropout_p > 0`` drops each probability with that chance (the mask is a
    function of ``seed`` and the element's batch, head, row and key) and
    scales the kept ones by 1 / (1 - dropout_p); LSE stays the undropped one.
    Dropout calls are not split and do not combine with ``window``.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError(f"unsupported dtype {q.dtype}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must have the same dtype")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, S, H, D] and k, v [B, S, H_kv, D]")
    if k.shape[0] != q.shape[0] or k.shape[1] != q.shape[1] or k.shape[3] != q.shape[3] or \
            k.shape[2] < 1 or q.shape[2] % k.shape[2] != 0:
        raise ValueError("k, v must match q in B, S, D, with H_kv dividing H")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    _check_devices(q.device, k=k, v=v, out=out, lse=lse)
    if not (0.0 <= dropout_p < 1.0):
        raise ValueError("dropout_p must be in [0, 1)")
    if dropout_p > 0.0 and window is not None:
        raise ValueError("dropout does not combine with a window")
    B, S, H, D = q.shape
    H_kv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None and with_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (B, H, S) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] tensor")
    dtype = FA_F16 if q.dtype == torch.float16 else FA_BF16
    with torch.cuda.device(q.device):
        st = _stream_handle(stream)
        lse_ptr = lse.data_ptr() if lse is not None else None
        nbytes = (fa_splitkv_workspace_size(B, H, S, D, causal)
                  if split_kv and window is None and dropout_p == 0.0 else 0)
        if dropout_p > 0.0:
            rc = fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                                B, H, H_kv, S, D, causal, dropout_p, seed, scale, dtype, st)
        elif window is not None:
            rc = fa_fwd_local(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                              B, H, H_kv, S, D, causal, int(window[0]), int(window[1]), scale,
                              dtype, st)
        elif nbytes > 0:
            ws = _workspace(q.device, st, nbytes)
            rc = fa_fwd_gqa_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse_ptr, B, H, H_kv, S, D, causal, scale, dtype, ws.data_ptr(),
                                    ws.numel(), st)
        else:
            rc = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                            B, H, H_kv, S, D, causal, scale, dtype, st)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse


def attention_forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                             scale: float | None = None, out=None, lse=None,
                             with_lse: bool = True, stream=None):
    """O, LSE of a packed variable-length batch of torch CUDA tensors.

    q [total, H, D], k, v [total, H_kv, D] (contiguous fp16 / bf16, H_kv
    dividing H), cu_seqlens an int32 CUDA tensor [B + 1] of sequence offsets
    (cu_seqlens[0] = 0), max_seqlen the longest sequence.  Returns
    out [total, H, D] and lse [H, total] (fp32); every tensor on q's device.
    Work is enqueued on ``stream`` (a torch stream or a raw handle; default:
    the current stream) and not waited for; offsets that are out of range are
    reported by ``fa_device_status()``.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens", cu_seqlens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must be fp16 or bf16 of one dtype")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be an int32 tensor [B + 1]")
    _check_devices(q.device, k=k, v=v, cu_seqlens=cu_seqlens, out=out, lse=lse)
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or k.shape[0] != q.shape[0] \
            or k.shape[2] != q.shape[2] or q.shape[1] % k.shape[1] != 0:
        raise ValueError("q must be [total, H, D] and k, v [total, H_kv, D], H_kv dividing H")
    total, H, D = q.shape
    H_kv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None and with_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (H, total) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [H, total] tensor")
    dtype = FA_F16 if q.dtype == torch.float16 else FA_BF16
    with torch.cuda.device(q.device):
        st = _stream_handle(stream)
        rc = fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, cu_seqlens.data_ptr(),
                           B, max_seqlen, total, H, H_kv, D, causal, scale, dtype, st)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return out, lse
