"""Pins of the backward-pass oracle.

The gradients are pinned to the forward definition itself by central finite
differences of L = sum(O * G) (G a fixed upstream gradient), and by closed
forms and invariants of softmax attention.  The real-valued forward used for
the differences is pinned to the storage-bits forward oracle.
Source: "CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 反向 (Backward).
"""
import numpy as np
import pytest

import oracle

NONE, CAUSAL = oracle.MASK_NONE, oracle.MASK_CAUSAL
QB, QE = oracle.QBEGIN, oracle.QEND


def rand(seed, B, Sq, Sk, H, D):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Sq, H, D)), r.standard_normal((B, Sk, H, D)),
            r.standard_normal((B, Sk, H, D)), r.standard_normal((B, Sq, H, D)))


@pytest.mark.parametrize("mask,ct,Sq,Sk", [(NONE, QB, 5, 7), (CAUSAL, QB, 6, 6), (CAUSAL, QB, 4, 7),
                                           (CAUSAL, QE, 7, 4), (CAUSAL, QE, 3, 8)])
def test_gradients_match_central_differences_of_the_forward(mask, ct, Sq, Sk):
    q, k, v, g = rand(Sq * 10 + Sk, 1, Sq, Sk, 2, 4)
    scale = 0.7

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd_f64(q_, k_, v_, scale, mask, ct)
        return float(np.sum(o * g))

    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, g, scale, mask, ct)
    eps = 1e-6
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = loss(q, k, v)
            x[idx] = old - eps
            lm = loss(q, k, v)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-8), np.abs(grad - num).max()


def test_real_valued_forward_matches_the_storage_forward():
    r = np.random.default_rng(3)
    enc = lambda x: oracle.encode(oracle.BF16, x)
    qb, kb, vb = enc(r.standard_normal((2, 9, 3, 16))), enc(r.standard_normal((2, 11, 3, 16))), \
        enc(r.standard_normal((2, 11, 3, 16)))
    for mask, ct in ((NONE, QB), (CAUSAL, QB), (CAUSAL, QE)):
        o_bits, lse_bits = oracle.fmha_fwd(qb, kb, vb, oracle.BF16, 2, 3, 3, 9, 11, 16, 0.3, 1.0, mask, ct)
        dec = lambda b: oracle.decode(oracle.BF16, b)
        o, lse = oracle.attn_fwd_f64(dec(qb), dec(kb), dec(vb), 0.3, mask, ct)
        # the storage oracle reports rows in LSE order (b, h, i)
        assert np.allclose(o.transpose(0, 2, 1, 3).reshape(-1, 16), o_bits, atol=1e-13)
        assert np.allclose(lse.reshape(-1), lse_bits, atol=1e-13)


def test_equal_keys_give_zero_query_gradient_and_mean_value_gradient():
    q, k, v, g = rand(4, 1, 6, 9, 2, 8)
    k[:] = k[:, :1]                           # every key of a head equal
    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, g, 0.4)
    assert np.abs(dq).max() < 1e-12
    # uniform attention: dV_j = mean over queries of dO (each row gives 1/Sk)
    assert np.allclose(dv, np.broadcast_to(g.sum(axis=1, keepdims=True) / 9, dv.shape), atol=1e-12)


@pytest.mark.parametrize("mask,ct", [(NONE, QB), (CAUSAL, QB), (CAUSAL, QE)])
def test_key_gradients_sum_to_zero(mask, ct):
    # each row of dS sums to zero, so sum_j dK_j = scale * sum_i q_i * 0
    q, k, v, g = rand(5, 2, 7, 10, 3, 8)
    _, dk, _ = oracle.attn_bwd_f64(q, k, v, g, 0.6, mask, ct)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12


def test_keys_no_query_sees_get_no_gradient():
    q, k, v, g = rand(6, 1, 4, 9, 2, 8)
    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, g, 0.5, CAUSAL, QB)   # keys 4..8 are after every query
    assert np.all(dk[:, 4:] == 0) and np.all(dv[:, 4:] == 0)
    assert np.abs(dk[:, :4]).max() > 0 and np.abs(dv[:, :4]).max() > 0
    # q-end with more queries than keys: the first rows see no key and get no gradient
    dq, _, _ = oracle.attn_bwd_f64(*rand(7, 1, 9, 4, 2, 8), 0.5, CAUSAL, QE)
    assert np.all(dq[:, :5] == 0) and np.abs(dq[:, 5:]).max() > 0


@pytest.mark.parametrize("mask,ct,Sq,Sk", [(NONE, QB, 5, 7), (CAUSAL, QB, 6, 6), (CAUSAL, QE, 7, 4)])
def test_given_o_backward_equals_the_definition_with_the_exact_o(mask, ct, Sq, Sk):
    # D_i = dO_i . O_i from the exact O is the same number as sum_j P_ij dP_ij
    q, k, v, g = rand(Sq * 7 + Sk, 2, Sq, Sk, 2, 4)
    o, _ = oracle.attn_fwd_f64(q, k, v, 0.6, mask, ct)
    for a, b in zip(oracle.attn_bwd_o_f64(q, k, v, o, g, 0.6, mask, ct), oracle.attn_bwd_f64(q, k, v, g, 0.6, mask, ct)):
        assert np.allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mask,ct,Sq,Sk", [(NONE, QB, 5, 7), (CAUSAL, QB, 6, 6), (CAUSAL, QE, 7, 4)])
def test_given_o_backward_responds_to_a_changed_o_by_the_closed_form(mask, ct, Sq, Sk):
    # O -> O + E changes D_i by c_i = dO_i . E_i, so dS_ij by -P_ij c_i:
    # dQ_i by -scale c_i sum_j P_ij K_j, dK_j by -scale sum_i P_ij c_i Q_i, dV not at all.
    # P comes from the forward oracle with unit-vector values (O = P exactly).
    B, H, D, scale = 1, 2, 4, 0.6
    q, k, v, g = rand(Sq * 3 + Sk, B, Sq, Sk, H, D)
    o, _ = oracle.attn_fwd_f64(q, k, v, scale, mask, ct)
    e = np.random.default_rng(5).standard_normal(o.shape)
    # P [B, Sq, H, Sk], D columns at a time: V_j = the unit vector e_(j - j0) for keys
    # j in [j0, j0 + D), 0 for the others, gives O = P[:, :, :, j0:j0 + D]
    p = np.zeros((B, Sq, H, Sk))
    for j0 in range(0, Sk, D):
        unit = np.zeros((B, Sk, H, D))
        for j in range(j0, min(j0 + D, Sk)):
            unit[:, j, :, j - j0] = 1.0
        pc, _ = oracle.attn_fwd_f64(q, k, unit, scale, mask, ct)
        p[..., j0:j0 + D] = pc[..., :min(D, Sk - j0)]
    c = np.sum(g * e, axis=-1)                                       # [B, Sq, H]
    dq0, dk0, dv0 = oracle.attn_bwd_o_f64(q, k, v, o, g, scale, mask, ct)
    dq1, dk1, dv1 = oracle.attn_bwd_o_f64(q, k, v, o + e, g, scale, mask, ct)
    want_dq = -scale * c[..., None] * np.einsum("bihj,bjhd->bihd", p, k)
    want_dk = -scale * np.einsum("bihj,bih,bihd->bjhd", p, c, q)
    assert np.allclose(dq1 - dq0, want_dq, rtol=0, atol=1e-12)
    assert np.allclose(dk1 - dk0, want_dk, rtol=0, atol=1e-12)
    assert np.array_equal(dv1, dv0)
