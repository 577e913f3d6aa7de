"""Work accounting for the attention forward pass (measurement, not compute).

The FLOP count is the two GEMMs of the definition, 2*Sq*Sk*D each per head,
i.e. 4*B*H*Sq*Sk*D, halved for a causal mask.  This is the accounting that the
"fmha sm120 : 超越 torch.sdpa(flash-attention-2)" page uses for its §3
benchmark table; a test reproduces that table's TFLOP/s column from its
millisecond column.
"""
from __future__ import annotations

from typing import Optional, Sequence


def attention_flops(B: int, H: int, Sq: int, Sk: int, D: int, causal: bool,
                    seqlens_q: Optional[Sequence[int]] = None,
                    seqlens_k: Optional[Sequence[int]] = None) -> float:
    """Algorithmic FLOPs of one forward call (varlen: summed per sequence)."""
    f = 0.5 if causal else 1.0
    if seqlens_q is not None:
        return sum(4.0 * H * lq * lk * D * f for lq, lk in zip(seqlens_q, seqlens_k))
    return 4.0 * B * H * Sq * Sk * D * f


def algorithmic_bytes(B: int, H: int, H_k: int, Sq: int, Sk: int, D: int, elem_bytes: int,
                      out_bytes: int, with_lse: bool = True,
                      seqlens_q: Optional[Sequence[int]] = None,
                      seqlens_k: Optional[Sequence[int]] = None) -> float:
    """Compulsory HBM traffic: Q, K, V read once, O (and fp32 LSE) written once."""
    if seqlens_q is not None:
        tq, tk = sum(seqlens_q), sum(seqlens_k)
    else:
        tq, tk = B * Sq, B * Sk
    rd = tq * H * D * elem_bytes + 2 * tk * H_k * D * elem_bytes
    wr = tq * H * D * out_bytes + (tq * H * 4 if with_lse else 0)
    return float(rd + wr)


def gen_bytes(B: int, H: int, H_k: int, seqlens: Sequence[int], insert: bool, elem_bytes: int,
              D: int = 128, with_lse: bool = True) -> float:
    """Algorithmic HBM bytes of one generation-phase call: every cached K and V
    row of the attended tokens read once, the new K/V rows read and written into
    the cache (insert mode), q read, O (and LSE) written."""
    rows = sum(int(L) for L in seqlens)
    kv = 2.0 * rows * H_k * D * elem_bytes
    new = (2.0 * 2.0 * B * H_k * D * elem_bytes) if insert else 0.0
    qo = 2.0 * B * H * D * elem_bytes
    return kv + new + qo + (4.0 * B * H if with_lse else 0.0)


def gen_flops(H: int, seqlens: Sequence[int], insert: bool, D: int = 128) -> float:
    """The two products of the definition for one query row per head: 4*D per key."""
    return sum(4.0 * H * (int(L) + (1 if insert else 0)) * D for L in seqlens)
