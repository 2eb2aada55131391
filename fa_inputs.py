"""Seeded synthetic inputs for the attention forward pass.

This module is the only code that both the fp64 oracle (``oracle/``) and the
CUDA path (``attention_forward_fwd_gb300``) see.  It draws random numbers,
casts them to the 16-bit storage type and arranges them in the contiguous
``[B, S, H, D]`` layout.  It holds none of the attention arithmetic.

Every tensor is returned as a numpy ``uint16`` array of IEEE binary16 or
bfloat16 bit patterns, so that the oracle can decode exactly the values the
GPU reads.  ``to_torch`` wraps such an array as a torch tensor of the matching
dtype without copying.

Workloads
---------
The five workloads are the ones the attention forward is measured on (the
FlashAttention-2 teaching case on page "CuTe 详解：以 FlashAttention-2 拆解
Layout、TiledCopy 与 TiledMMA", sections 教学配置 and 正确性、编译与计时方法):

=========  ==================================================================
name       shape / values
=========  ==================================================================
s256       B=1,H=1,S=256,D=64 fp16, Q,K,V iid N(0,1), scale 1/8, non-causal
s4096      B=1,H=1,S=4096,D=64 fp16, iid N(0,1), scale 1/8, both masks
b4h16      B=4,H=16,S=4096,D=64 fp16, iid N(0,1), scale 1/8, causal
b2h16d128  B=2,H=16,S=8192,D=128 bf16, iid N(0,1), scale 1/sqrt(128), both
stress     B=3,H=8,S=1999,D=64 fp16, Q,K = 4*N(0,1), V ~ U[-1,1], scale 1/8,
           both masks; head (b=2,h=7) has every key equal to key 0
=========  ==================================================================

Seeds are ``1000 + index`` (index 1..5 in the order above).  A sixth workload,
b4h32kv8d128 (B=4, 32 query heads over 8 K/V heads, S=4096, D=128 bf16,
causal, seed 1006), measures grouped K/V heads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_qkv", "make_qkv_for", "to_torch",
           "f32_to_bits", "attention_flops", "make_varlen", "varlen_lengths"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str            # "f16" or "bf16"
    dist: str             # "normal" or "stress"
    scale: float
    modes: tuple          # causal flags the workload is run with
    seed: int
    identical_key_head: tuple = field(default=())   # (b, h) or ()
    h_kv: int | None = None   # K/V heads when grouped (query heads share them)

    @property
    def kv_heads(self) -> int:
        return self.H if self.h_kv is None else self.h_kv


WORKLOADS = {
    "s256": Workload("s256", 1, 1, 256, 64, "f16", "normal", 1.0 / 8.0,
                     (False,), 1001),
    "s4096": Workload("s4096", 1, 1, 4096, 64, "f16", "normal", 1.0 / 8.0,
                      (False, True), 1002),
    "b4h16": Workload("b4h16", 4, 16, 4096, 64, "f16", "normal", 1.0 / 8.0,
                      (True,), 1003),
    "b2h16d128": Workload("b2h16d128", 2, 16, 8192, 128, "bf16", "normal",
                          1.0 / math.sqrt(128.0), (True, False), 1004),
    "stress": Workload("stress", 3, 8, 1999, 64, "f16", "stress", 1.0 / 8.0,
                       (True, False), 1005, identical_key_head=(2, 7)),
    # grouped K/V heads (GQA): 32 query heads sharing 8 K/V heads, the
    # production extension beyond the five configurations
    "b4h32kv8d128": Workload("b4h32kv8d128", 4, 32, 4096, 128, "bf16", "normal",
                             1.0 / math.sqrt(128.0), (True,), 1006, h_kv=8),
}


def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the 16-bit storage type (round to nearest
    even) and return the bit patterns as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch  # the cast is torch's; nothing of the method is here
        t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
        return t.numpy().view(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def make_qkv(B: int, H: int, S: int, D: int, dtype: str = "f16",
             dist: str = "normal", seed: int = 0,
             identical_key_head: tuple = (), h_kv: int | None = None):
    """Draw Q, K, V as uint16 bit arrays of shape [B, S, H, D].

    dist="normal": Q, K, V iid N(0, 1).
    dist="stress": Q, K = 4 * N(0, 1) (peaky softmax), V ~ U[-1, 1].
    identical_key_head=(b, h): every key row of that head is set to its row 0.
    h_kv: K and V get h_kv heads ([B, S, h_kv, D]) instead of H.
    """
    rng = np.random.default_rng(seed)
    shape = (B, S, H, D)
    kv_shape = shape if h_kv is None else (B, S, h_kv, D)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(kv_shape, dtype=np.float32)
    if dist == "normal":
        v = rng.standard_normal(kv_shape, dtype=np.float32)
    elif dist == "stress":
        q *= 4.0
        k *= 4.0
        v = rng.uniform(-1.0, 1.0, size=kv_shape).astype(np.float32)
    else:
        raise ValueError(f"unknown dist {dist!r}")
    if identical_key_head:
        b, h = identical_key_head
        k[b, :, h, :] = k[b, 0, h, :]
    return (f32_to_bits(q, dtype), f32_to_bits(k, dtype), f32_to_bits(v, dtype))


def make_varlen(seqlens, H: int, D: int, dtype: str = "f16", dist: str = "normal",
                seed: int = 0, h_kv: int | None = None):
    """Packed variable-length batch: Q [total, H, D] and K, V [total, h_kv, D]
    as uint16 bit arrays (sequence b is rows cu[b] .. cu[b+1]-1), and the
    int32 offsets cu = [0, S_0, S_0 + S_1, ...] (length B + 1)."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    total = int(cu[-1])
    q, k, v = make_qkv(1, H, total, D, dtype, dist, seed, h_kv=h_kv)
    return q[0], k[0], v[0], cu


def varlen_lengths(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """B sequence lengths drawn uniformly from [lo, hi] (a mixed-length batch)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=B)


def make_qkv_for(w: Workload):
    return make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.dist, w.seed,
                    w.identical_key_head, h_kv=w.h_kv)


def to_torch(bits: np.ndarray, dtype: str):
    """View a uint16 bit array as a CPU torch tensor of dtype f16/bf16."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def attention_flops(B: int, H: int, S: int, D: int, causal: bool) -> float:
    """Counted FLOPs of one forward: 4*B*H*S^2*D, half of it when causal."""
    f = 4.0 * B * H * S * S * D
    return f / 2.0 if causal else f
