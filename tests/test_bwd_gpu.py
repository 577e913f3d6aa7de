"""Backward pass (fmha_bwd) against the oracle, on the GPU.

The forward kernel supplies O and LSE, as in training; the oracle recomputes
everything exactly from the stored inputs.  The kernel rounds P and dS to the
input type for the tensor cores and each gradient to the output type, so an
element may differ from the exact gradient by 1% of that gradient's largest
magnitude plus half a unit in the last place of the output (relative error of a
16-bit P or dS term: 2^-9; sums over up to a few thousand terms).

e4m3 inputs (with O as the e4m3 forward writes it) are widened exactly to bf16
and take bf16 gradients; they are compared with the oracle's backward that
forms the row sums of O * dO from that stored O, on the decoded inputs, under
the same bf16 bound.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import half_ulp

pytestmark = pytest.mark.gpu

DT = {"bf16": (torch.bfloat16, oracle.BF16), "f16": (torch.float16, oracle.F16)}
MASK = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL}
CT = {"qbegin": oracle.QBEGIN, "qend": oracle.QEND}


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


def run_case_e4m3(fm, B, H, Sq, Sk, D, mask, ct, seed):
    g = torch.Generator().manual_seed(seed)
    e4 = lambda *s: torch.randn(*s, generator=g).clamp_(-448, 448).to(torch.float8_e4m3fn)
    q, k, v, do = e4(B, Sq, H, D), e4(B, Sk, H, D), e4(B, Sk, H, D), e4(B, Sq, H, D)
    dev = "cuda"
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = fm.fwd(qd, kd, vd, mask=mask, causal_type=ct)
    assert o.dtype == torch.float8_e4m3fn
    dq, dk, dv = fm.bwd(qd, kd, vd, o, dod, lse, mask=mask, causal_type=ct)
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    assert dq.dtype == dk.dtype == dv.dtype == torch.bfloat16
    dec = lambda t: oracle.decode(oracle.E4M3, t.cpu().view(torch.uint8).numpy())
    ref = oracle.attn_bwd_o_f64(dec(q), dec(k), dec(v), dec(o), dec(do), D ** -0.5, MASK[mask], CT[ct])
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        got = got.float().cpu().numpy().astype(np.float64)
        assert not np.isnan(got).any(), f"NaN in {name}"
        scale = np.abs(want).max() if want.size else 0.0
        bound = 1e-2 * scale + half_ulp("bf16", want)
        err = np.abs(got - want)
        assert (err <= bound).all(), (f"{name}: worst {err.max():.4g} (scale {scale:.3g}) at "
                                      f"{np.unravel_index(err.argmax(), err.shape)}")
        assert err.mean() <= 2e-3 * max(scale, 1e-6), (name, err.mean(), scale)


E4M3_CASES = [
    # B, H, Sq, Sk, D, mask, causal_type
    (1, 2, 128, 128, 128, "none", "qbegin"),
    (2, 3, 300, 300, 128, "causal", "qbegin"),
    (1, 4, 200, 333, 64, "none", "qbegin"),
    (2, 2, 257, 129, 128, "causal", "qend"),
    (2, 16, 2048, 2048, 128, "causal", "qbegin"),     # more work units than SMs
]


@pytest.mark.parametrize("case", E4M3_CASES, ids=[f"e4m3_b{c[0]}h{c[1]}_{c[2]}x{c[3]}_d{c[4]}_{c[5]}_{c[6]}"
                                                  for c in E4M3_CASES])
def test_bwd_e4m3_matches_oracle(fm, case):
    run_case_e4m3(fm, *case, seed=sum(case[:5]) + 1)


def run_case(fm, dtype, B, H, Sq, Sk, D, mask, ct, seed):
    tdt, odt = DT[dtype]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Sq, H, D, generator=g).to(tdt)
    k = torch.randn(B, Sk, H, D, generator=g).to(tdt)
    v = torch.randn(B, Sk, H, D, generator=g).to(tdt)
    do = torch.randn(B, Sq, H, D, generator=g).to(tdt)
    dev = "cuda"
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = fm.fwd(qd, kd, vd, mask=mask, causal_type=ct)
    dq, dk, dv = fm.bwd(qd, kd, vd, o, dod, lse, mask=mask, causal_type=ct)
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    dec = lambda t: oracle.decode(odt, t.view(torch.uint16).numpy())
    ref = oracle.attn_bwd_f64(dec(q), dec(k), dec(v), dec(do), D ** -0.5, MASK[mask], CT[ct])
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        got = got.float().cpu().numpy().astype(np.float64)
        assert not np.isnan(got).any(), f"NaN in {name}"
        scale = np.abs(want).max() if want.size else 0.0
        bound = 1e-2 * scale + half_ulp(dtype, want)
        err = np.abs(got - want)
        assert (err <= bound).all(), (f"{name}: worst {err.max():.4g} (scale {scale:.3g}) at "
                                      f"{np.unravel_index(err.argmax(), err.shape)}")
        assert err.mean() <= 2e-3 * max(scale, 1e-6), (name, err.mean(), scale)


CASES = [
    # dtype, B, H, Sq, Sk, D, mask, causal_type
    ("bf16", 1, 2, 128, 128, 128, "none", "qbegin"),
    ("bf16", 2, 3, 300, 300, 128, "causal", "qbegin"),
    ("f16", 1, 4, 200, 333, 64, "none", "qbegin"),
    ("bf16", 2, 2, 257, 129, 128, "causal", "qend"),
    ("f16", 1, 2, 130, 400, 128, "causal", "qend"),
    ("bf16", 1, 2, 96, 700, 64, "causal", "qbegin"),     # keys after every query get zero gradient
    ("bf16", 2, 4, 1024, 1024, 128, "causal", "qbegin"),
    # more work units than SMs: each CTA runs several (b, h, tile) units in
    # turn, reusing its accumulators, ring slots and barrier phases
    ("bf16", 2, 16, 2048, 2048, 128, "causal", "qbegin"),
    ("f16", 1, 20, 1536, 1536, 64, "none", "qbegin"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_b{c[1]}h{c[2]}_{c[3]}x{c[4]}_d{c[5]}_{c[6]}_{c[7]}"
                                             for c in CASES])
def test_bwd_matches_oracle(fm, case):
    run_case(fm, *case, seed=sum(case[1:6]))


def test_bwd_empty_sides_give_zero(fm):
    k = torch.randn(1, 64, 2, 64, device="cuda", dtype=torch.bfloat16)
    q = torch.empty(1, 0, 2, 64, device="cuda", dtype=torch.bfloat16)
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(k, 3.0)
    lse = torch.empty(1, 2, 0, device="cuda")
    fm.bwd(q, k, k, q, q, lse, dk=dk, dv=dv, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())


@pytest.mark.parametrize("b,h", [(0, 0), (1, 15)])
def test_bwd_full_size_sampled_heads(fm, b, h):
    """The benchmark's backward workload at full size (causal B=2 H=16 S=8192
    D=128 bf16, the launch bench.py times); heads are independent, so the
    oracle checks every gradient element of sampled (batch, head) pairs."""
    B, H, S, D = 2, 16, 8192, 128
    g = torch.Generator().manual_seed(1234)
    q, k, v, do = (torch.randn(B, S, H, D, generator=g).to(torch.bfloat16) for _ in range(4))
    dev = "cuda"
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = fm.fwd(qd, kd, vd, mask="causal")
    dq, dk, dv = fm.bwd(qd, kd, vd, o, dod, lse, mask="causal")
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    dec = lambda t: oracle.decode(oracle.BF16, t[b:b + 1, :, h:h + 1].contiguous().view(torch.uint16).numpy())
    ref = oracle.attn_bwd_f64(dec(q), dec(k), dec(v), dec(do), D ** -0.5, oracle.MASK_CAUSAL, oracle.QBEGIN)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        got = got[b:b + 1, :, h:h + 1].float().cpu().numpy().astype(np.float64)
        assert not np.isnan(got).any(), f"NaN in {name}"
        scale = np.abs(want).max()
        bound = 1e-2 * scale + half_ulp("bf16", want)
        err = np.abs(got - want)
        assert (err <= bound).all(), (f"{name}: worst {err.max():.4g} (scale {scale:.3g}) at "
                                      f"{np.unravel_index(err.argmax(), err.shape)}")
        assert err.mean() <= 2e-3 * max(scale, 1e-6), (name, err.mean(), scale)
