"""Helpers for the GPU parity tests: run the library on an Inputs bundle with
guard bands around every output, and compare with the oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

from head_attention_forward_02_gb300 import workloads as wl
from tests.helpers import oracle_on

GUARD = 4096           # guard elements on each side of O (keeps 16-byte alignment)
SENTINEL = 0x7F        # byte pattern written into every guard and padding region
TOL_O = {"f16": 1e-2, "bf16": 1e-2, "e4m3": 6e-2}
TOL_LSE = 1e-3
MANT = {"f16": (10, -14), "bf16": (7, -126), "e4m3": (3, -6)}


def half_ulp(dtype: str, x: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of the output type at |x|."""
    mbits, emin = MANT[dtype]
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, emin)
    return 0.5 * np.exp2(e - mbits)


class Run:
    """One library call with guarded outputs; holds host copies of the results."""

    def __init__(self, fm, inp: wl.Inputs, impl: str = "tc", lse: bool = True, num_splits=None):
        w = inp.w
        dev = torch.device("cuda")
        self.inp = inp
        tdt = wl.DTYPES[w.dtype]
        esz = torch.empty((), dtype=tdt).element_size()
        if inp.cu_seqlens_q is not None:
            T, pad = inp.total_length, inp.pad_rows
            q_full = inp.q_full.to(dev)
            k_full = inp.k_full.to(dev)
            v_full = inp.v_full.to(dev)
            q, k, v = q_full[pad:], k_full[pad:], v_full[pad:]
            o_rows = pad + T
            o_elems = o_rows * w.H * w.D
            self.o_buf = torch.full(((GUARD * 2 + o_elems) * esz,), SENTINEL, dtype=torch.uint8,
                                    device=dev)
            o_all = self.o_buf[GUARD * esz: GUARD * esz + o_elems * esz].view(tdt).view(o_rows, w.H, w.D)
            o = o_all[pad:]
            n_lse = w.H * T
            cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
            B = len(inp.seqlens_q)
            kw = dict(cu_seqlens_q=cq, cu_seqlens_k=ck, max_len=inp.max_len, total_length=T)
        else:
            q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
            o_elems = q.numel()
            self.o_buf = torch.full(((GUARD * 2 + o_elems) * esz,), SENTINEL, dtype=torch.uint8,
                                    device=dev)
            o = self.o_buf[GUARD * esz: GUARD * esz + o_elems * esz].view(tdt).view(q.shape)
            n_lse = w.B * w.H * w.Sq
            kw = {}
        self.lse_buf = torch.full(((GUARD * 2 + n_lse) * 4,), SENTINEL, dtype=torch.uint8, device=dev)
        lse_t = self.lse_buf[GUARD * 4: GUARD * 4 + n_lse * 4].view(torch.float32)
        fm.fwd(q, k, v, scale=w.softmax_scale, out_scale=w.out_scale, mask=w.mask,
               causal_type=w.causal_type, out=o, lse=lse_t if lse else None, return_lse=lse,
               impl=impl, num_splits=num_splits, **kw)
        torch.cuda.synchronize()
        self.status = fm.device_status(reset=True)
        self.esz = esz
        self.o = o
        self.lse = lse_t
        self.has_lse = lse

    def guards_intact(self) -> bool:
        e = self.esz
        ob = self.o_buf
        ok = bool((ob[:GUARD * e] == SENTINEL).all()) and bool((ob[-GUARD * e:] == SENTINEL).all())
        lb = self.lse_buf
        ok = ok and bool((lb[:GUARD * 4] == SENTINEL).all()) and bool((lb[-GUARD * 4:] == SENTINEL).all())
        inp = self.inp
        if inp.cu_seqlens_q is not None:
            # leading padding batch and rows past the last sequence stay untouched
            pad = inp.pad_rows * inp.w.H * inp.w.D * e
            ok = ok and bool((ob[GUARD * e: GUARD * e + pad] == SENTINEL).all())
            end = int(inp.cu_seqlens_q[-1])
            T = inp.total_length
            if end < T:
                o_rows = self.o.view(torch.uint8).view(T, -1)
                ok = ok and bool((o_rows[end:] == SENTINEL).all())
                if self.has_lse:
                    l2 = self.lse.view(torch.uint8).view(inp.w.H, T, 4)
                    ok = ok and bool((l2[:, end:] == SENTINEL).all())
            if not self.has_lse:
                ok = ok and bool((self.lse_buf == SENTINEL).all())
        elif not self.has_lse:
            ok = ok and bool((self.lse_buf == SENTINEL).all())
        return ok

    def rows(self, rows: np.ndarray):
        """O (float64 [n, D]) and LSE (float64 [n]) at oracle row indices."""
        inp, w = self.inp, self.inp.w
        rows = torch.from_numpy(np.asarray(rows, dtype=np.int64))
        if inp.cu_seqlens_q is not None:
            T = inp.total_length
            h, t = rows // T, rows % T
            o = self.o[t.cuda(), h.cuda()]
        else:
            b = rows // (w.H * w.Sq)
            h = (rows // w.Sq) % w.H
            i = rows % w.Sq
            o = self.o[b.cuda(), i.cuda(), h.cuda()]
        lse = self.lse[rows.cuda()] if self.has_lse else None
        o = o.to(torch.float64).cpu().numpy()
        lse = lse.to(torch.float64).cpu().numpy() if lse is not None else None
        return o, lse


def all_rows(inp: wl.Inputs) -> np.ndarray:
    w = inp.w
    if inp.cu_seqlens_q is not None:
        end = int(inp.cu_seqlens_q[-1])
        T = inp.total_length
        return np.array([h * T + t for h in range(w.H) for t in range(end)], dtype=np.int64)
    return np.arange(w.B * w.H * w.Sq, dtype=np.int64)


def sample_rows(inp: wl.Inputs, n: int, seed: int) -> np.ndarray:
    """Heads 0 and H-1 at tile edges plus a seeded uniform sample."""
    w = inp.w
    rng = np.random.default_rng(seed)
    if inp.cu_seqlens_q is not None:
        T = inp.total_length
        cq = inp.cu_seqlens_q.tolist()
        toks = set()
        for b in range(len(cq) - 1):
            for e in (0, 127, 128, 255, 256):
                if cq[b] + e < cq[b + 1]:
                    toks.add(cq[b] + e)
            if cq[b + 1] > cq[b]:
                toks.add(cq[b + 1] - 1)
        base = [h * T + t for h in (0, w.H - 1) for t in sorted(toks)]
        extra = rng.choice(all_rows(inp), size=n, replace=False)
    else:
        edges = [e for e in (0, 1, 127, 128, 255, 256, w.Sq // 2, w.Sq - 129, w.Sq - 128, w.Sq - 1)
                 if 0 <= e < w.Sq]
        base = [(b * w.H + h) * w.Sq + i for b in (0, w.B - 1) for h in (0, w.H - 1) for i in edges]
        extra = rng.integers(0, w.B * w.H * w.Sq, size=n)
    return np.unique(np.concatenate([np.array(base, dtype=np.int64), extra.astype(np.int64)]))


def e4m3_weight_bound(oracle, inp: wl.Inputs, rows: np.ndarray, threads: int = 0) -> np.ndarray:
    """Worst-case effect on O of rounding the attention weights P to e4m3 before
    the P.V product: every weight in e4m3's normal range is off by at most 2^-4
    of itself (3 mantissa bits, round to nearest even), and the row sum l is
    taken from the unrounded weights, so |dO| <= 2^-4 * out_scale * sum_j p_j
    |v_j| / l -- the attention output of |V|, which the oracle computes exactly
    (|x| of an e4m3 value is an e4m3 value)."""
    v_abs = inp.v.float().abs().to(inp.v.dtype)
    absv = wl.Inputs(inp.w, inp.q, inp.k, v_abs, cu_seqlens_q=inp.cu_seqlens_q,
                     cu_seqlens_k=inp.cu_seqlens_k, seqlens_q=inp.seqlens_q, seqlens_k=inp.seqlens_k,
                     total_length=inp.total_length, max_len=inp.max_len, pad_rows=inp.pad_rows)
    o_abs, _ = oracle_on(oracle, absv, rows=rows, threads=threads)
    return 2.0 ** -4 * np.abs(o_abs)


def compare(run: Run, oracle, rows: np.ndarray, threads: int = 0, extra=None) -> dict:
    """Check O and LSE at the given rows against the oracle; returns error stats.
    ``extra`` (an array shaped like O's rows) widens the O bound element by
    element where a derived rounding term applies."""
    w = run.inp.w
    o_ref, lse_ref = oracle_on(oracle, run.inp, rows=rows, threads=threads)
    o, lse = run.rows(rows)
    err = np.abs(o - o_ref)
    bound = TOL_O[w.dtype] + half_ulp(w.dtype, o_ref)
    if extra is not None:
        bound = bound + extra
    bad = err > bound
    stats = {"max_err": float(err.max()) if err.size else 0.0,
             "mean_err": float(err.mean()) if err.size else 0.0,
             "n_rows": int(rows.size)}
    assert not np.isnan(o).any(), "NaN in O"
    assert not bad.any(), (
        f"O mismatch at {int(bad.sum())} elements; worst err {err.max():.4g} "
        f"(bound there {bound.flat[err.argmax()]:.4g}) row {rows[np.argwhere(bad)[0][0]]}")
    if lse is not None:
        masked = np.isneginf(lse_ref)
        assert np.all(np.isneginf(lse[masked])), "fully masked rows must give LSE = -inf"
        assert np.all(o[masked] == 0), "fully masked rows must give O = 0"
        d = np.abs(lse[~masked] - lse_ref[~masked])
        stats["lse_max_err"] = float(d.max()) if d.size else 0.0
        assert not np.isnan(lse).any()
        assert (d <= TOL_LSE).all(), f"LSE mismatch, worst {d.max():.4g}"
    # the mean bound carries the mean of the same output-rounding term as the
    # per-element bound: rounding O to the output type is part of every
    # element's error (large |O| in peaked rows), it does not average out
    mean_tol = (1e-3 if w.dtype != "e4m3" else 1e-2) + float(np.mean(half_ulp(w.dtype, o_ref)))
    if extra is not None:
        mean_tol += float(np.mean(extra))
    assert stats["mean_err"] <= mean_tol, stats
    return stats
