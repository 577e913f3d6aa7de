"""Python binding of the C ABI in include/fmha.h (argument marshalling only).

Every step of the computation runs in libfmha.so's CUDA kernels; this module
only turns torch tensors into pointers and the current torch stream into a
cudaStream_t.  If the library has not been built it raises: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfmha.so")

F16, BF16, E4M3 = 0, 1, 2
MASK_NONE, MASK_RESIDUAL, MASK_CAUSAL = 0, 1, 2
CAUSAL_QBEGIN, CAUSAL_QEND = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4

_TORCH_DTYPE = {torch.float16: F16, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}
_MASKS = {"none": MASK_NONE, "residual": MASK_RESIDUAL, "causal": MASK_CAUSAL}
_CAUSAL = {"qbegin": CAUSAL_QBEGIN, "qend": CAUSAL_QEND}

EXPORTED = ("fmha_fwd", "fmha_fwd_simt", "fmha_fwd_splitkv", "fmha_fwd_splitkv_workspace_size",
            "fmha_fwd_splitkv_noalloc",
            "fmha_status_string", "fmha_device_status", "fmha_kv_tile_range")


class fmha_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int)]


class FmhaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load libfmha.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(_LIB_PATH)
        fwd_args = [fmha_tensor, fmha_tensor, fmha_tensor, fmha_tensor, ctypes.c_void_p,
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                    ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                    ctypes.c_void_p]
        for name in ("fmha_fwd", "fmha_fwd_simt"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = fwd_args
        L.fmha_fwd_splitkv.restype = ctypes.c_int
        L.fmha_fwd_splitkv.argtypes = fwd_args[:-1] + [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                                       ctypes.c_void_p]
        L.fmha_fwd_splitkv_noalloc.restype = ctypes.c_int
        L.fmha_fwd_splitkv_noalloc.argtypes = fwd_args[:-1] + [ctypes.c_int, ctypes.c_void_p]
        L.fmha_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
        L.fmha_fwd_splitkv_workspace_size.argtypes = [ctypes.c_int] * 5 + [ctypes.c_int64]
        L.fmha_gen_fwd.restype = ctypes.c_int
        L.fmha_gen_fwd.argtypes = [fmha_tensor] * 6 + [ctypes.c_void_p] + [ctypes.c_int] * 6 + [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_float, ctypes.c_void_p,
            ctypes.c_size_t, ctypes.c_void_p]
        L.fmha_gen_workspace_size.restype = ctypes.c_size_t
        L.fmha_gen_workspace_size.argtypes = [ctypes.c_int] * 5
        L.fmha_bwd.restype = ctypes.c_int
        L.fmha_bwd.argtypes = [fmha_tensor] * 5 + [ctypes.c_void_p] + [fmha_tensor] * 3 + [ctypes.c_int] * 5 + [
            ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.fmha_bwd_workspace_size.restype = ctypes.c_size_t
        L.fmha_bwd_workspace_size.argtypes = [ctypes.c_int] * 3
        L.fmha_bwd_workspace_size_ex.restype = ctypes.c_size_t
        L.fmha_bwd_workspace_size_ex.argtypes = [ctypes.c_int] * 6
        L.fmha_status_string.restype = ctypes.c_char_p
        L.fmha_status_string.argtypes = [ctypes.c_int]
        L.fmha_device_status.restype = ctypes.c_int
        L.fmha_device_status.argtypes = [ctypes.c_int]
        L.fmha_set_wait_limit_ns.restype = ctypes.c_int
        L.fmha_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.fmha_set_test_gate.restype = ctypes.c_int
        L.fmha_set_test_gate.argtypes = [ctypes.c_int]
        L.fmha_kv_tile_range.restype = ctypes.c_int
        L.fmha_kv_tile_range.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int)] * 2
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fmha_status_string(int(status)).decode()


def device_status(reset: bool = False) -> int:
    return lib().fmha_device_status(1 if reset else 0)


def set_wait_limit_ns(ns: int) -> int:
    """Test hook (see fmha_set_wait_limit_ns): the forward kernels' bounded waits
    give up after ns nanoseconds; 0 restores the default."""
    return lib().fmha_set_wait_limit_ns(int(ns))


def set_test_gate(on: bool) -> int:
    """Test hook (see fmha_set_test_gate): the forward's producer first waits for
    a flag that nothing sets."""
    return lib().fmha_set_test_gate(1 if on else 0)


def kv_tile_range(q_row0: int, q_rows: int, Sq: int, Sk: int, mask: int, causal_type: int,
                  tile_n: int) -> Tuple[int, int]:
    a, b = ctypes.c_int(), ctypes.c_int()
    rc = lib().fmha_kv_tile_range(q_row0, q_rows, Sq, Sk, mask, causal_type, tile_n,
                                  ctypes.byref(a), ctypes.byref(b))
    if rc != OK:
        raise FmhaError(rc, status_string(rc))
    return a.value, b.value


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _tensor(t, dtype: Optional[int] = None) -> fmha_tensor:
    if t is None:
        return fmha_tensor(None, BF16 if dtype is None else dtype)
    if isinstance(t, torch.Tensor):
        return fmha_tensor(t.data_ptr(), _TORCH_DTYPE[t.dtype] if dtype is None else dtype)
    return fmha_tensor(int(t), dtype)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _call(name, q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask, causal_type,
          cu_seqlens_q, cu_seqlens_k, max_len, total_length, stream) -> int:
    f = getattr(lib(), name)
    return f(_tensor(q), _tensor(k), _tensor(v), _tensor(o), _ptr(lse), int(B), int(H), int(H_k),
             int(Sq), int(Sk), int(D), float(scale), float(out_scale), int(mask), int(causal_type),
             _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_len), int(total_length),
             _stream(stream))


def fmha_fwd(q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask, causal_type,
             cu_seqlens_q=None, cu_seqlens_k=None, max_len=0, total_length=0, stream=None) -> int:
    """Same arguments, order and status codes as the C function fmha_fwd.

    Tensors are passed as torch tensors (or raw device addresses); ``stream``
    defaults to torch's current stream.  Returns the C status code."""
    return _call("fmha_fwd", q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                 causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length, stream)


def fmha_fwd_simt(q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask, causal_type,
                  cu_seqlens_q=None, cu_seqlens_k=None, max_len=0, total_length=0,
                  stream=None) -> int:
    """The CUDA-core cross-check kernel; same contract as fmha_fwd."""
    return _call("fmha_fwd_simt", q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                 causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length, stream)


def fmha_fwd_splitkv(q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask, causal_type,
                     cu_seqlens_q=None, cu_seqlens_k=None, max_len=0, total_length=0,
                     num_splits=1, workspace=None, workspace_bytes=None, stream=None) -> int:
    """Same arguments, order and status codes as the C function fmha_fwd_splitkv."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().fmha_fwd_splitkv(
        _tensor(q), _tensor(k), _tensor(v), _tensor(o), _ptr(lse), int(B), int(H), int(H_k), int(Sq),
        int(Sk), int(D), float(scale), float(out_scale), int(mask), int(causal_type),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_len), int(total_length), int(num_splits),
        _ptr(workspace), int(workspace_bytes), _stream(stream))


def fmha_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                             causal_type, cu_seqlens_q=None, cu_seqlens_k=None, max_len=0,
                             total_length=0, num_splits=1, stream=None) -> int:
    """Same arguments, order and status codes as the C function
    fmha_fwd_splitkv_noalloc: split-KV with the library's built-in scratch,
    for callers that must not allocate device memory while they run."""
    return lib().fmha_fwd_splitkv_noalloc(
        _tensor(q), _tensor(k), _tensor(v), _tensor(o), _ptr(lse), int(B), int(H), int(H_k), int(Sq),
        int(Sk), int(D), float(scale), float(out_scale), int(mask), int(causal_type),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_len), int(total_length), int(num_splits),
        _stream(stream))


def fmha_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits, total_length=0) -> int:
    return int(lib().fmha_fwd_splitkv_workspace_size(int(B), int(H), int(Sq), int(D), int(num_splits),
                                                     int(total_length)))


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
        out_scale: float = 1.0, mask: str = "none", causal_type: str = "qbegin",
        cu_seqlens_q: Optional[torch.Tensor] = None, cu_seqlens_k: Optional[torch.Tensor] = None,
        max_len: Optional[int] = None, total_length: Optional[int] = None,
        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
        return_lse: bool = True, impl: str = "tc", num_splits: Optional[int] = None, stream=None):
    """Attention forward on device tensors; allocates O (and LSE) if not given.

    Fixed length: q [B,Sq,H,D], k/v [B,Sk,H_k,D].  Varlen: q [T,H,D], k/v
    [T,H_k,D] with int32 device cumulative lengths.  ``num_splits`` selects
    the split-KV entry point (a workspace is allocated with torch).
    Returns (O, LSE)."""
    varlen = cu_seqlens_q is not None
    D = q.shape[-1]
    if varlen:
        T = q.shape[0] if total_length is None else int(total_length)
        B = cu_seqlens_q.numel() - 1
        H, H_k = q.shape[1], k.shape[1]
        Sq = Sk = 0
        if max_len is None:
            raise ValueError("varlen needs max_len")
        lse_shape = (H, T)
    else:
        B, Sq, H = q.shape[0], q.shape[1], q.shape[2]
        Sk, H_k = k.shape[1], k.shape[2]
        T = 0
        lse_shape = (B, H, Sq)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    if num_splits is not None:
        nbytes = fmha_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits, T)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        rc = fmha_fwd_splitkv(q, k, v, out, lse, B, H, H_k, Sq, Sk, D, sc, out_scale, _MASKS[mask],
                              _CAUSAL[causal_type], cu_seqlens_q, cu_seqlens_k, max_len or 0, T,
                              num_splits, ws, nbytes, stream)
        if rc != OK:
            raise FmhaError(rc, status_string(rc))
        return out, lse
    name = "fmha_fwd" if impl == "tc" else "fmha_fwd_simt"
    rc = _call(name, q, k, v, out, lse, B, H, H_k, Sq, Sk, D, sc, out_scale, _MASKS[mask],
               _CAUSAL[causal_type], cu_seqlens_q, cu_seqlens_k, max_len or 0, T, stream)
    if rc != OK:
        raise FmhaError(rc, status_string(rc))
    return out, lse


def fmha_gen_fwd(q, k_cache, v_cache, k_new, v_new, o, lse, B, H, H_k, D, B_cache, S_max, seqlen,
                 batch_idx, scale, out_scale, workspace, workspace_bytes, stream=None) -> int:
    """Same arguments, order and status codes as the C function fmha_gen_fwd."""
    dt = _TORCH_DTYPE[q.dtype] if isinstance(q, torch.Tensor) else None
    return lib().fmha_gen_fwd(
        _tensor(q), _tensor(k_cache), _tensor(v_cache), _tensor(k_new, dt), _tensor(v_new, dt), _tensor(o),
        _ptr(lse), int(B), int(H), int(H_k), int(D), int(B_cache), int(S_max), _ptr(seqlen),
        _ptr(batch_idx), float(scale), float(out_scale), _ptr(workspace), int(workspace_bytes),
        _stream(stream))


def fmha_gen_workspace_size(B, H, H_k, D, S_max) -> int:
    return int(lib().fmha_gen_workspace_size(int(B), int(H), int(H_k), int(D), int(S_max)))


def gen_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlen: torch.Tensor, *,
            k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
            batch_idx: Optional[torch.Tensor] = None, scale: Optional[float] = None,
            out_scale: float = 1.0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            return_lse: bool = True, workspace: Optional[torch.Tensor] = None, stream=None):
    """Generation-phase attention on device tensors (see fmha_gen_fwd).

    q [B, H, 128]; k_cache / v_cache [B_cache, S_max, H_k, 128]; seqlen int32
    [B]; k_new / v_new [B, H_k, 128] (insert mode) or None (cache-only);
    batch_idx int32 [B] or None.  Allocates O, LSE and the workspace with torch
    when not given.  Returns (O, LSE)."""
    B, H, D = q.shape
    B_cache, S_max, H_k = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    nbytes = fmha_gen_workspace_size(B, H, H_k, D, S_max) if B > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    rc = fmha_gen_fwd(q, k_cache, v_cache, k_new, v_new, out, lse, B, H, H_k, D, B_cache, S_max, seqlen,
                      batch_idx, sc, out_scale, workspace, max(nbytes, workspace.numel()), stream)
    if rc != OK:
        raise FmhaError(rc, status_string(rc))
    return out, lse


def fmha_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, scale, mask, causal_type, workspace,
             workspace_bytes, stream=None) -> int:
    """Same arguments, order and status codes as the C function fmha_bwd."""
    return lib().fmha_bwd(_tensor(q), _tensor(k), _tensor(v), _tensor(o), _tensor(dout), _ptr(lse), _tensor(dq),
                          _tensor(dk), _tensor(dv), int(B), int(H), int(Sq), int(Sk), int(D), float(scale),
                          int(mask), int(causal_type), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fmha_bwd_workspace_size(B, H, Sq) -> int:
    return int(lib().fmha_bwd_workspace_size(int(B), int(H), int(Sq)))


def fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, dtype) -> int:
    return int(lib().fmha_bwd_workspace_size_ex(int(B), int(H), int(Sq), int(Sk), int(D), int(dtype)))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
        lse: torch.Tensor, *, scale: Optional[float] = None, mask: str = "none", causal_type: str = "qbegin",
        dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
        workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of fwd (see fmha_bwd): q, o, dout [B,Sq,H,D]; k, v [B,Sk,H,D];
    lse [B,H,Sq] from fwd.  Allocates the gradients (bf16 for e4m3 inputs, else
    the inputs' type) and the workspace with torch when not given.  Returns
    (dq, dk, dv)."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    gdt = torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype
    dq = torch.empty(q.shape, dtype=gdt, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=gdt, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=gdt, device=v.device) if dv is None else dv
    nbytes = fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, _TORCH_DTYPE[q.dtype])
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    rc = fmha_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, sc, _MASKS[mask], _CAUSAL[causal_type],
                  workspace, max(nbytes, workspace.numel()), stream)
    if rc != OK:
        raise FmhaError(rc, status_string(rc))
    return dq, dk, dv
