"""The C-ABI library builds, loads and exports every declared symbol, and
rejects bad arguments before touching the GPU.  No compute call is made."""
import ctypes
import os
import re

import pytest

import attention_forward_fwd_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.library()


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert set(fa.EXPORTED_SYMBOLS) <= set(names), names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    texts = [fa.fa_status_string(code) for code in range(7)]
    assert all(texts) and len(set(texts)) == 7 and "unknown status" not in texts
    assert fa.fa_status_string(fa.FA_ERR_DEVICE_CHECK).startswith("a device-side invariant check")
    assert fa.fa_status_string(99) == "unknown status"


def test_last_device_status_is_exported_with_a_stream_argument(lib):
    """The stream-ordered status read takes one stream handle (no GPU call
    here: only its presence and signature in the header)."""
    import re
    with open(os.path.join(ROOT, "include", "fa_gb300.h")) as f:
        text = f.read()
    assert re.search(r"int\s+fa_last_device_status\s*\(\s*fa_stream_t\s+stream\s*\)", text)
    assert "fa_last_device_status" in fa.EXPORTED_SYMBOLS
    assert lib.fa_last_device_status.argtypes == [ctypes.c_void_p]


GOOD = dict(Q=4096, K=8192, V=12288, O=16384, LSE=20480, B=1, H=1, S=128, D=64,
            causal=0, scale=0.125, dtype=fa.FA_F16, stream=None)


@pytest.mark.parametrize("change,status", [
    (dict(Q=None), fa.FA_ERR_INVALID_ARG),
    (dict(K=None), fa.FA_ERR_INVALID_ARG),
    (dict(V=None), fa.FA_ERR_INVALID_ARG),
    (dict(O=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(S=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(D=100), fa.FA_ERR_UNSUPPORTED),   # not a multiple of 8
    (dict(D=264), fa.FA_ERR_UNSUPPORTED),   # above 256
    (dict(D=512), fa.FA_ERR_UNSUPPORTED),
    (dict(D=4), fa.FA_ERR_UNSUPPORTED),
    (dict(D=0), fa.FA_ERR_UNSUPPORTED),
    (dict(Q=4096 + 8), fa.FA_ERR_UNSUPPORTED),
    (dict(O=16384 + 2), fa.FA_ERR_UNSUPPORTED),
    (dict(LSE=20480 + 2), fa.FA_ERR_UNSUPPORTED),
    (dict(S=256 * 65535 + 1), fa.FA_ERR_UNSUPPORTED),
])
def test_bad_arguments_are_rejected_before_launch(lib, change, status):
    args = dict(GOOD, **change)
    rc = fa.fa_fwd(args["Q"], args["K"], args["V"], args["O"], args["LSE"], args["B"],
                   args["H"], args["S"], args["D"], args["causal"], args["scale"],
                   args["dtype"], args["stream"])
    assert rc == status


def test_dtype_specific_entry_points_validate(lib):
    assert fa.fa_fwd_f16(None, 1, 1, 1, None, 1, 1, 1, 64, 0, 1.0, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_bf16(16, 16, 16, 16, None, 1, 1, 1, 84, 0, 1.0, None) == fa.FA_ERR_UNSUPPORTED


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 8, 1, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.attention_forward(q, q, q)


def test_splitkv_entry_points_validate_before_cuda(lib):
    import ctypes
    assert lib.fa_splitkv_workspace_size(1, 1, 128, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.fa_splitkv_workspace_size(1, 1, 128, 84, 0, ctypes.byref(n)) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_splitkv_workspace_size(0, 1, 128, 64, 0, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_splitkv_launches(1, 1, 0, 64, 0) == 0
    bad = fa.fa_fwd_splitkv(None, 16, 16, 16, None, 1, 1, 128, 64, 0, 0.125, fa.FA_F16,
                            None, 0, None)
    assert bad == fa.FA_ERR_INVALID_ARG
    bad = fa.fa_fwd_splitkv(16, 16, 16, 16, None, 1, 1, 128, 100, 0, 0.125, fa.FA_F16,
                            None, 0, None)
    assert bad == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("H,H_kv", [(4, 0), (4, -1), (4, 3), (6, 4), (1, 2)])
def test_gqa_entry_points_reject_bad_group_before_cuda(lib, H, H_kv):
    """H_kv must be >= 1 and divide H; checked before anything is launched."""
    args = (16, 16, 16, 16, None, 1, H, H_kv, 128, 64, 0, 0.125, fa.FA_F16)
    assert fa.fa_fwd_gqa(*args, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_gqa_splitkv(*args, None, 0, None) == fa.FA_ERR_INVALID_ARG


def test_gqa_entry_points_validate_like_fa_fwd(lib):
    assert fa.fa_fwd_gqa(None, 16, 16, 16, None, 1, 4, 2, 128, 64, 0, 0.125, fa.FA_F16, None) \
        == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_gqa(16, 16, 16, 16, None, 1, 4, 2, 128, 100, 0, 0.125, fa.FA_F16, None) \
        == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_gqa(16, 16, 24, 16, None, 1, 4, 2, 128, 64, 0, 0.125, fa.FA_F16, None) \
        == fa.FA_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_binding_rejects_mismatched_kv_heads():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs CUDA tensors to get past the device check")
    q = torch.zeros(1, 8, 4, 64, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, 8, 3, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        fa.attention_forward(q, k, k)


def test_binding_takes_torch_stream_objects_and_raw_handles():
    class FakeStream:
        cuda_stream = 0x1234
    assert fa._stream_handle(FakeStream()) == 0x1234
    assert fa._stream_handle(0x5678) == 0x5678


def test_binding_rejects_tensors_on_another_device():
    import torch
    here, there = torch.device("cuda", 0), torch.device("cuda", 1)

    class T:
        def __init__(self, dev):
            self.device = dev
    fa._check_devices(here, k=T(here), v=T(here), out=None, lse=None)
    for name in ("k", "v", "out", "lse", "cu_seqlens"):
        tensors = dict(k=T(here), v=T(here))
        tensors[name] = T(there)
        with pytest.raises(ValueError, match=name):
            fa._check_devices(here, **tensors)
