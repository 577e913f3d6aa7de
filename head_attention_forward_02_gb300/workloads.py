"""Seeded synthetic inputs for the attention forward pass.

This module only draws and packs random numbers; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle take their inputs
from here, so that they see the same stored values.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
as N(0, 1) in float32 and then cast to the storage type (fp8 e4m3 inputs are
clamped to +-448 first, the largest finite e4m3 value).  Variable-length
workloads are packed back to back after one leading padding batch of
``max_len`` rows, the layout the CUTLASS Blackwell FMHA walkthrough asks for
(§变长序列: "valid but never used" padding ahead of the first batch).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
# codes shared with the C ABI (include/fmha.h) -- plain enum values, no arithmetic
DTYPE_CODE = {"f16": 0, "bf16": 1, "e4m3": 2}
MASK_CODE = {"none": 0, "residual": 1, "causal": 2}
CAUSAL_CODE = {"qbegin": 0, "qend": 1}
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    dtype: str = "bf16"
    B: int = 1
    H: int = 1
    H_k: int = 1
    Sq: int = 128
    Sk: int = 128
    D: int = 128
    mask: str = "none"
    causal_type: str = "qbegin"
    scale: Optional[float] = None          # None -> 1/sqrt(D)
    out_scale: float = 1.0
    seqlens_q: Optional[List[int]] = None  # varlen when both are given
    seqlens_k: Optional[List[int]] = None
    seed: int = 0
    # varlen: draw this many lengths uniform in [lo, hi] (inclusive) from the seed
    varlen_draw: Optional[tuple] = None

    @property
    def varlen(self) -> bool:
        return self.seqlens_q is not None or self.varlen_draw is not None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)


@dataclass
class Inputs:
    """Host tensors for one call.  For varlen the real data of each packed tensor
    starts after ``pad_rows`` padding rows: ``q_full[pad_rows:]`` is what the
    kernel sees."""
    w: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_full: Optional[torch.Tensor] = None
    k_full: Optional[torch.Tensor] = None
    v_full: Optional[torch.Tensor] = None
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_k: Optional[torch.Tensor] = None
    seqlens_q: Optional[List[int]] = None
    seqlens_k: Optional[List[int]] = None
    total_length: int = 0
    max_len: int = 0
    pad_rows: int = 0


def _randn(shape, gen, dtype: str) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if dtype == "e4m3":
        x = x.clamp_(-E4M3_MAX, E4M3_MAX)
    return x.to(DTYPES[dtype])


def _cumsum(lens: List[int]) -> torch.Tensor:
    out = [0]
    for n in lens:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def generate(w: Workload, seed: Optional[int] = None) -> Inputs:
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    if not w.varlen:
        q = _randn((w.B, w.Sq, w.H, w.D), gen, w.dtype)
        k = _randn((w.B, w.Sk, w.H_k, w.D), gen, w.dtype)
        v = _randn((w.B, w.Sk, w.H_k, w.D), gen, w.dtype)
        return Inputs(w, q, k, v)
    if w.varlen_draw is not None:
        n, lo, hi = w.varlen_draw
        lens = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
        lq, lk = list(lens), list(lens)
    else:
        lq, lk = list(w.seqlens_q), list(w.seqlens_k)
    assert len(lq) == len(lk)
    cq, ck = _cumsum(lq), _cumsum(lk)
    total = max(int(cq[-1]), int(ck[-1]), 1)
    max_len = max([1] + lq + lk)
    pad = max_len
    q_full = _randn((pad + total, w.H, w.D), gen, w.dtype)
    k_full = _randn((pad + total, w.H_k, w.D), gen, w.dtype)
    v_full = _randn((pad + total, w.H_k, w.D), gen, w.dtype)
    return Inputs(w, q_full[pad:], k_full[pad:], v_full[pad:], q_full, k_full, v_full,
                  cq, ck, lq, lk, total, max_len, pad)


def bits(t: torch.Tensor):
    """Raw storage bits of a tensor as a numpy array (uint16, or uint8 for fp8)."""
    t = t.contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view("uint16")


# The five workloads the benchmark and the parity tests are built around.
CONFIGS = {
    "fp16_b1_h2_s128_d64_nomask": Workload(
        "fp16_b1_h2_s128_d64_nomask", dtype="f16", B=1, H=2, H_k=2, Sq=128, Sk=128, D=64,
        mask="none", seed=1),
    "bf16_causal_b4_h16_s2048_d128": Workload(
        "bf16_causal_b4_h16_s2048_d128", dtype="bf16", B=4, H=16, H_k=16, Sq=2048, Sk=2048,
        D=128, mask="causal", causal_type="qbegin", seed=2),
    "bf16_causal_gqa_b2_h32_hk8_s8192_d128": Workload(
        "bf16_causal_gqa_b2_h32_hk8_s8192_d128", dtype="bf16", B=2, H=32, H_k=8, Sq=8192,
        Sk=8192, D=128, mask="causal", causal_type="qbegin", seed=3),
    "bf16_varlen_causal_8x_u256_4096_h16_d128": Workload(
        "bf16_varlen_causal_8x_u256_4096_h16_d128", dtype="bf16", B=8, H=16, H_k=16, D=128,
        mask="causal", causal_type="qbegin", varlen_draw=(8, 256, 4096), seed=4),
    "e4m3_nomask_b1_h16_s16384_d128": Workload(
        "e4m3_nomask_b1_h16_s16384_d128", dtype="e4m3", B=1, H=16, H_k=16, Sq=16384,
        Sk=16384, D=128, mask="none", out_scale=1.0, seed=5),
}

# More shapes of the same forward kernel, timed next to the five above: other
# head dims, the unmasked and long causal cases and causal e4m3.  Each has a
# many-unit parity test at the same sizes (tests/test_shapes_gpu.py).
EXTRA_CONFIGS = {
    w.name: w for w in [
        Workload("bf16_causal_b8_h16_s4096_d64", dtype="bf16", B=8, H=16, H_k=16, Sq=4096, Sk=4096, D=64,
                 mask="causal", seed=6),
        Workload("bf16_causal_b4_h16_s4096_d32", dtype="bf16", B=4, H=16, H_k=16, Sq=4096, Sk=4096, D=32,
                 mask="causal", seed=7),
        Workload("bf16_nomask_gqa_b2_h32_hk8_s8192_d128", dtype="bf16", B=2, H=32, H_k=8, Sq=8192, Sk=8192,
                 D=128, mask="none", seed=8),
        Workload("bf16_causal_b1_h32_s16384_d128", dtype="bf16", B=1, H=32, H_k=32, Sq=16384, Sk=16384,
                 D=128, mask="causal", seed=9),
        Workload("e4m3_causal_gqa_b2_h32_hk8_s8192_d128", dtype="e4m3", B=2, H=32, H_k=8, Sq=8192, Sk=8192,
                 D=128, mask="causal", seed=10),
        Workload("e4m3_causal_b4_h16_s4096_d64", dtype="e4m3", B=4, H=16, H_k=16, Sq=4096, Sk=4096, D=64,
                 mask="causal", seed=11),
    ]
}


# ----------------------------------------------------------------------------
# Generation phase: one new query token per sequence against a K/V cache
# ----------------------------------------------------------------------------

@dataclass
class GenWorkload:
    name: str
    dtype: str = "bf16"
    B: int = 1
    H: int = 32
    H_k: int = 8
    S_max: int = 8192
    lengths: str = "full"          # "full": S_max - 1 cached tokens; "uniform": U[S_max/8, S_max-1]
    insert: bool = True            # new K/V row written into the cache and attended
    seed: int = 1


@dataclass
class GenInputs:
    w: GenWorkload
    q: torch.Tensor                # [B, H, 128]
    k_cache: torch.Tensor          # [B, S_max, H_k, 128]
    v_cache: torch.Tensor
    k_new: Optional[torch.Tensor]  # [B, H_k, 128] or None (cache-only)
    v_new: Optional[torch.Tensor]
    seqlen: torch.Tensor           # int32 [B]


def generate_gen(w: GenWorkload, seed: Optional[int] = None) -> GenInputs:
    """Seeded N(0,1) query, caches and new rows; every cache row is finite."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    D = 128
    q = _randn((w.B, w.H, D), gen, w.dtype)
    kc = _randn((w.B, w.S_max, w.H_k, D), gen, w.dtype)
    vc = _randn((w.B, w.S_max, w.H_k, D), gen, w.dtype)
    kn = _randn((w.B, w.H_k, D), gen, w.dtype) if w.insert else None
    vn = _randn((w.B, w.H_k, D), gen, w.dtype) if w.insert else None
    top = w.S_max - (1 if w.insert else 0)
    if w.lengths == "full":
        sl = torch.full((w.B,), top, dtype=torch.int32)
    else:
        sl = torch.randint(max(1, w.S_max // 8), top + 1, (w.B,), generator=gen, dtype=torch.int32)
    return GenInputs(w, q, kc, vc, kn, vn, sl)


GEN_CONFIGS = {
    "gen_bf16_b32_h32_hk8_s8192": GenWorkload("gen_bf16_b32_h32_hk8_s8192", B=32, H=32, H_k=8, S_max=8192,
                                              lengths="full", seed=21),
    "gen_bf16_varlen_b64_h32_hk8_s16384": GenWorkload("gen_bf16_varlen_b64_h32_hk8_s16384", B=64, H=32, H_k=8,
                                                      S_max=16384, lengths="uniform", seed=22),
    "gen_f16_b8_h64_hk2_s32768_cacheonly": GenWorkload("gen_f16_b8_h64_hk2_s32768_cacheonly", dtype="f16", B=8,
                                                       H=64, H_k=2, S_max=32768, lengths="full", insert=False,
                                                       seed=23),
    "gen_e4m3_b32_h32_hk8_s8192": GenWorkload("gen_e4m3_b32_h32_hk8_s8192", dtype="e4m3", B=32, H=32, H_k=8,
                                              S_max=8192, lengths="full", seed=24),
}
