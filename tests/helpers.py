"""Shared test helpers: tensor <-> raw-bit conversion and oracle calls on Inputs."""
from __future__ import annotations

import numpy as np
import torch

from head_attention_forward_02_gb300 import workloads as wl

ORACLE_DTYPE = {"f16": 0, "bf16": 1, "e4m3": 2}


def exact(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a stored tensor, through torch's own widening
    conversion (independent of the oracle's bit decoders)."""
    return t.to(torch.float64).numpy()


def oracle_on(oracle, inp: wl.Inputs, rows=None, threads=0, mask=None, causal_type=None,
              out_scale=None, scale=None):
    """Run the oracle on an Inputs bundle; returns (O [n, D], LSE [n])."""
    w = inp.w
    m = wl.MASK_CODE[mask or w.mask]
    ct = wl.CAUSAL_CODE[causal_type or w.causal_type]
    sc = w.softmax_scale if scale is None else scale
    osc = w.out_scale if out_scale is None else out_scale
    if inp.cu_seqlens_q is not None:
        return oracle.fmha_fwd(wl.bits(inp.q), wl.bits(inp.k), wl.bits(inp.v), ORACLE_DTYPE[w.dtype],
                               len(inp.seqlens_q), w.H, w.H_k, 0, 0, w.D, sc, osc, m, ct,
                               inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(),
                               inp.total_length, rows=rows, threads=threads)
    return oracle.fmha_fwd(wl.bits(inp.q), wl.bits(inp.k), wl.bits(inp.v), ORACLE_DTYPE[w.dtype],
                           w.B, w.H, w.H_k, w.Sq, w.Sk, w.D, sc, osc, m, ct,
                           rows=rows, threads=threads)


def fixed_inputs(dtype="bf16", B=1, H=2, H_k=2, Sq=16, Sk=16, D=8, mask="none",
                 causal_type="qbegin", seed=0, out_scale=1.0, scale=None) -> wl.Inputs:
    w = wl.Workload("t", dtype=dtype, B=B, H=H, H_k=H_k, Sq=Sq, Sk=Sk, D=D, mask=mask,
                    causal_type=causal_type, seed=seed, out_scale=out_scale, scale=scale)
    return wl.generate(w)


def varlen_inputs(lq, lk, dtype="bf16", H=2, H_k=2, D=8, mask="none", causal_type="qbegin",
                  seed=0) -> wl.Inputs:
    w = wl.Workload("t", dtype=dtype, H=H, H_k=H_k, D=D, mask=mask, causal_type=causal_type,
                    seqlens_q=list(lq), seqlens_k=list(lk), seed=seed)
    return wl.generate(w)
