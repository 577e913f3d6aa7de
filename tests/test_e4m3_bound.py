"""CPU check of the derived e4m3 bound for peaked attention.

With e4m3 inputs the tensor-core kernel rounds the attention weights P to e4m3
before the P.V product, relative to a reference maximum that may lag the true
row maximum by up to 2^8 (lazy rescaling), and divides by the sum of the
unrounded weights.  tests.gpu_util.e4m3_weight_bound states the worst case of
that rounding as 2^-4 * (attention output of |V|).  Here a plain numpy model of
exactly that rounding (float64 scores, weights against a randomly stale
reference maximum, torch's e4m3 cast) is run on peaked inputs, and its error
against the oracle must stay inside 6e-2 + the derived term -- the bound the
GPU test asserts.  The model is test code, not the kernel.
"""
import numpy as np
import torch

from tests.gpu_util import TOL_O, all_rows, e4m3_weight_bound
from tests.helpers import fixed_inputs, oracle_on


def _peaked_inputs():
    inp = fixed_inputs(dtype="e4m3", B=1, H=2, H_k=1, Sq=300, Sk=420, D=128, mask="none", seed=31)
    gain = torch.ones(420)
    gain[:128], gain[128:256], gain[256:] = 0.1, 2.0, 6.0
    inp.k[:] = (inp.k.float() * gain[None, :, None, None]).to(inp.k.dtype)
    return inp


def _model(inp, rng):
    """O with P rounded to e4m3 against a stale reference max (rows in oracle order)."""
    w = inp.w
    q = inp.q.double().numpy()[0]          # [Sq, H, D]
    k = inp.k.double().numpy()[0]          # [Sk, H_k, D]
    v = inp.v.double().numpy()[0]
    out = []
    for h in range(w.H):
        g = h // (w.H // w.H_k)
        s = (q[:, h, :] @ k[:, g, :].T) * w.softmax_scale * np.log2(np.e)     # log2 units
        m = s.max(axis=1, keepdims=True)
        m_ref = m - 8.0 * rng.random((s.shape[0], 1))                        # lag in [0, 8)
        p = np.exp2(s - m_ref)                                               # <= 256
        p_q = torch.from_numpy(p).to(torch.float8_e4m3fn).double().numpy()
        out.append((p_q @ v[:, g, :]) / p.sum(axis=1, keepdims=True))
    return np.concatenate(out, axis=0)


def test_derived_e4m3_bound_covers_the_weight_rounding(oracle):
    inp = _peaked_inputs()
    rows = all_rows(inp)
    o_ref, _ = oracle_on(oracle, inp, rows=rows)
    extra = e4m3_weight_bound(oracle, inp, rows)
    rng = np.random.default_rng(0)
    worst_plain, worst = 0.0, 0.0
    for _ in range(4):
        err = np.abs(_model(inp, rng) - o_ref)
        worst_plain = max(worst_plain, float(err.max()))
        worst = max(worst, float((err - extra).max()))
        assert (err <= TOL_O["e4m3"] + extra).all()
    # the case is a real one: the rounding alone breaks the plain e4m3 tolerance
    assert worst_plain > TOL_O["e4m3"]


def test_derived_term_is_the_weighted_mean_of_abs_v(oracle):
    # one visible key per row (causal q-begin, row 0) -> the term is 2^-4 |v_0|
    inp = fixed_inputs(dtype="e4m3", B=1, H=1, H_k=1, Sq=4, Sk=4, D=32, mask="causal", seed=3)
    extra = e4m3_weight_bound(oracle, inp, np.array([0]))
    np.testing.assert_allclose(extra[0], 2.0 ** -4 * np.abs(inp.v.double().numpy()[0, 0, 0]))
