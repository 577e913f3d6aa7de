"""CPU oracle for the fused attention forward pass (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference arm may import it.  The CUDA library
never loads it, and it never loads the CUDA library: the two share no code.

The arithmetic lives in ``fmha_oracle.c`` (plain C, double precision, OpenMP over
output rows).  It takes the raw storage bits of Q, K and V and decodes them with
its own decoders, so that it does not depend on any conversion routine used on
the CUDA side.  See the header of ``fmha_oracle.c`` for the definition it
computes and the passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fmha_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

F16, BF16, E4M3 = 0, 1, 2
MASK_NONE, MASK_RESIDUAL, MASK_CAUSAL = 0, 1, 2
QBEGIN, QEND = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into an in-tree shared object (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_decode.restype = ctypes.c_double
        lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
        lib.oracle_encode.restype = ctypes.c_uint32
        lib.oracle_encode.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.oracle_decode_array.restype = None
        lib.oracle_decode_array.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p]
        lib.oracle_encode_array.restype = None
        lib.oracle_encode_array.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p]
        lib.oracle_fmha_fwd.restype = ctypes.c_int
        lib.oracle_fmha_fwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_gen_fwd.restype = ctypes.c_int
        lib.oracle_gen_fwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_attn_fwd_f64.restype = ctypes.c_int
        lib.oracle_attn_fwd_f64.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_attn_bwd_f64.restype = ctypes.c_int
        lib.oracle_attn_bwd_f64.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int]
        lib.oracle_attn_bwd_o_f64.restype = ctypes.c_int
        lib.oracle_attn_bwd_o_f64.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int]
        _lib = lib
    return _lib


def _bits_dtype(dtype: int):
    return np.uint8 if dtype == E4M3 else np.uint16


def decode(dtype: int, bits: np.ndarray) -> np.ndarray:
    """Exact value (float64) of each stored code."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=_bits_dtype(dtype))
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_decode_array(dtype, b.ctypes.data, b.size, out.ctypes.data)
    return out


def encode(dtype: int, x: np.ndarray) -> np.ndarray:
    """Round float64 values to the storage type (nearest, ties to even)."""
    lib = _load()
    xx = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xx.shape, dtype=_bits_dtype(dtype))
    lib.oracle_encode_array(dtype, xx.ctypes.data, xx.size, out.ctypes.data)
    return out


def fmha_fwd(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, dtype: int,
             B: int, H: int, H_k: int, Sq: int, Sk: int, D: int,
             scale: float, out_scale: float = 1.0, mask: int = MASK_NONE,
             causal_type: int = QBEGIN,
             cu_seqlens_q: Optional[np.ndarray] = None,
             cu_seqlens_k: Optional[np.ndarray] = None,
             total_length: int = 0,
             rows: Optional[np.ndarray] = None,
             threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O (float64, before output rounding) and LSE (float64) for the selected rows.

    Layouts: fixed length q [B,Sq,H,D], k/v [B,Sk,H_k,D]; varlen q [total,H,D],
    k/v [total,H_k,D] with int32 cumulative lengths of B+1 entries.  Row indices
    follow the LSE layout: (b*H + h)*Sq + i, or h*total + t for varlen.
    ``rows=None`` returns every row.  Returns (O [n_rows, D], LSE [n_rows]).
    """
    lib = _load()
    bd = _bits_dtype(dtype)
    q = np.ascontiguousarray(q_bits, dtype=bd)
    k = np.ascontiguousarray(k_bits, dtype=bd)
    v = np.ascontiguousarray(v_bits, dtype=bd)
    varlen = cu_seqlens_q is not None and cu_seqlens_k is not None
    if varlen:
        cq = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        ck = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
        n_all = H * int(total_length)
    else:
        cq = ck = None
        n_all = B * H * Sq
    if rows is None:
        r = None
        n = n_all
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n = r.size
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_fmha_fwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype,
        B, H, H_k, Sq, Sk, D, float(scale), float(out_scale), mask, causal_type,
        cq.ctypes.data if varlen else None, ck.ctypes.data if varlen else None,
        int(total_length), r.ctypes.data if r is not None else None, n,
        o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def gen_fwd(q_bits: np.ndarray, k_cache_bits: np.ndarray, v_cache_bits: np.ndarray,
            k_new_bits: Optional[np.ndarray], v_new_bits: Optional[np.ndarray], dtype: int,
            B: int, H: int, H_k: int, D: int, B_cache: int, S_max: int,
            seqlen: np.ndarray, batch_idx: Optional[np.ndarray],
            scale: float, out_scale: float = 1.0, threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Generation phase: O (float64 [B*H, D], row b*H + h) and LSE (float64 [B*H]).

    q [B, H, D]; caches [B_cache, S_max, H_k, D]; new K/V [B, H_k, D] or None for
    cache-only; seqlen int32 [B] cached tokens per sequence; batch_idx int32 [B]
    (cache entry of sequence b) or None for the identity.  See ``oracle_gen_fwd``
    in ``fmha_oracle.c`` for the definition.
    """
    lib = _load()
    bd = _bits_dtype(dtype)
    arr = [np.ascontiguousarray(x, dtype=bd) if x is not None else None
           for x in (q_bits, k_cache_bits, v_cache_bits, k_new_bits, v_new_bits)]
    sl = np.ascontiguousarray(seqlen, dtype=np.int32)
    bi = np.ascontiguousarray(batch_idx, dtype=np.int32) if batch_idx is not None else None
    o = np.empty((B * H, D), dtype=np.float64)
    lse = np.empty((B * H,), dtype=np.float64)
    ptr = [a.ctypes.data if a is not None else None for a in arr]
    rc = lib.oracle_gen_fwd(*ptr, dtype, B, H, H_k, D, B_cache, S_max, sl.ctypes.data,
                            bi.ctypes.data if bi is not None else None, float(scale),
                            float(out_scale), o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def attn_fwd_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, mask: int = MASK_NONE,
                 causal_type: int = QBEGIN) -> Tuple[np.ndarray, np.ndarray]:
    """Forward on real values: q [B,Sq,H,D], k/v [B,Sk,H,D] (float64) -> O [B,Sq,H,D], LSE [B,H,Sq]."""
    lib = _load()
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    o = np.empty_like(q)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    if lib.oracle_attn_fwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Sq, Sk, D, float(scale),
                               mask, causal_type, o.ctypes.data, lse.ctypes.data) != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def attn_bwd_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, scale: float,
                 mask: int = MASK_NONE, causal_type: int = QBEGIN, threads: int = 0):
    """Backward on real values: (dQ, dK, dV) for upstream gradient dout [B,Sq,H,D].
    See ``oracle_attn_bwd_f64`` in ``fmha_oracle.c`` for the definition."""
    lib = _load()
    q, k, v, g = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    if lib.oracle_attn_bwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, B, H, Sq, Sk, D,
                               float(scale), mask, causal_type, dq.ctypes.data, dk.ctypes.data,
                               dv.ctypes.data, int(threads)) != 0:
        raise ValueError("oracle rejected the arguments")
    return dq, dk, dv


def attn_bwd_o_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, dout: np.ndarray, scale: float,
                   mask: int = MASK_NONE, causal_type: int = QBEGIN, threads: int = 0):
    """Backward with D_i = dO_i . O_i formed from the given O [B,Sq,H,D] (the row sums of
    O * dO).  See ``oracle_attn_bwd_o_f64`` in ``fmha_oracle.c``."""
    lib = _load()
    q, k, v, o, g = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, o, dout))
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    if lib.oracle_attn_bwd_o_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data, g.ctypes.data, B,
                                 H, Sq, Sk, D, float(scale), mask, causal_type, dq.ctypes.data,
                                 dk.ctypes.data, dv.ctypes.data, int(threads)) != 0:
        raise ValueError("oracle rejected the arguments")
    return dq, dk, dv
