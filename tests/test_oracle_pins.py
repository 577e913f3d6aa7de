"""Pins for the CPU oracle: closed forms, invariants and exact special cases.

None of these re-types the oracle's own formula.  Each checks the oracle
against something fixed independently -- a library decoder, a closed-form
answer, an invariance of the definition, or a brute force that takes a
different route (no max shift, exact summation) on tiny inputs -- chosen so
that a dropped term, a wrong sign, a wrong index or a transposed operand fails
at least one test.
"""
import math

import numpy as np
import pytest
import torch

from head_attention_forward_02_gb300 import workloads as wl
from tests.helpers import exact, fixed_inputs, oracle_on, varlen_inputs

# ----------------------------------------------------------------------------
# storage-format decoders and encoders
# ----------------------------------------------------------------------------


def _check_same(got, want):
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_f16_every_code(oracle):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    _check_same(oracle.decode(oracle.F16, codes), codes.view(np.float16).astype(np.float64))


def test_decode_bf16_every_code(oracle):
    # bfloat16 is the top half of an IEEE binary32 word
    codes = np.arange(65536, dtype=np.uint32)
    want = (codes << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    _check_same(oracle.decode(oracle.BF16, codes.astype(np.uint16)), want)


def test_decode_e4m3_every_code(oracle):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    _check_same(oracle.decode(oracle.E4M3, codes), want)
    d = oracle.decode(oracle.E4M3, np.array([0x7E, 0x38, 0x01, 0x08, 0x7F, 0xFF, 0x80], np.uint8))
    assert d[0] == 448.0 and d[1] == 1.0 and d[2] == 2.0 ** -9 and d[3] == 2.0 ** -6
    assert np.isnan(d[4]) and np.isnan(d[5]) and d[6] == 0.0 and np.signbit(d[6])


@pytest.mark.parametrize("dt,nb", [(0, 65536), (1, 65536), (2, 256)])
def test_encode_inverts_decode(oracle, dt, nb):
    codes = np.arange(nb, dtype=np.uint32).astype(np.uint8 if nb == 256 else np.uint16)
    vals = oracle.decode(dt, codes)
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.encode(dt, vals[ok]), codes[ok])


def test_encode_f16_round_nearest_even(oracle):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 5, 20000),
                        [2049.0, 2051.0, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 65519.0, 65520.0, 1e6]])
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode(oracle.F16, x), want)


def test_encode_bf16_round_nearest_even(oracle):
    rng = np.random.default_rng(1)
    x32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.encode(oracle.BF16, x32.astype(np.float64)), want)
    # ties: halfway cases go to the even mantissa
    t = oracle.encode(oracle.BF16, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8]))
    assert t[0] == 0x3F80 and t[1] == 0x3F82


def test_encode_e4m3_round_nearest_even_and_saturate(oracle):
    rng = np.random.default_rng(2)
    x32 = (rng.standard_normal(20000) * 2.0 ** rng.integers(-10, 8, 20000)).astype(np.float32)
    x32 = np.clip(x32, -448, 448)
    want = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode(oracle.E4M3, x32.astype(np.float64)), want)
    s = oracle.encode(oracle.E4M3, np.array([449.0, 470.0, 1e9, -1e9]))
    assert list(s) == [0x7E, 0x7E, 0x7E, 0xFE]


# ----------------------------------------------------------------------------
# attention: closed forms
# ----------------------------------------------------------------------------

def _allowed(mask, causal_type, i, sq, sk):
    if mask != "causal":
        return list(range(sk))
    off = sk - sq if causal_type == "qend" else 0
    return [j for j in range(sk) if j <= i + off]


@pytest.mark.parametrize("mask,ct,Sq,Sk", [("none", "qbegin", 9, 13), ("causal", "qbegin", 13, 13),
                                           ("causal", "qend", 7, 12), ("causal", "qend", 12, 7),
                                           ("causal", "qbegin", 12, 7)])
def test_uniform_keys_give_mean_of_visible_values(oracle, mask, ct, Sq, Sk):
    """All keys equal: every visible score is the same s, so O is the plain mean
    of the visible V rows (times out_scale) and LSE = s + ln(count)."""
    inp = fixed_inputs(B=2, H=4, H_k=2, Sq=Sq, Sk=Sk, D=8, mask=mask, causal_type=ct, seed=11,
                       out_scale=1.5)
    inp.k[:] = inp.k[:, :1].clone()
    o, lse = oracle_on(oracle, inp)
    Q, K, V = exact(inp.q), exact(inp.k), exact(inp.v)
    sc = inp.w.softmax_scale
    o = o.reshape(2, 4, Sq, 8)
    lse = lse.reshape(2, 4, Sq)
    for b in range(2):
        for h in range(4):
            g = h // 2
            for i in range(Sq):
                vis = _allowed(mask, ct, i, Sq, Sk)
                if not vis:
                    assert np.all(o[b, h, i] == 0) and lse[b, h, i] == -np.inf
                    continue
                s = sc * float(np.dot(Q[b, i, h], K[b, 0, g]))
                np.testing.assert_allclose(o[b, h, i], 1.5 * V[b, vis, g].mean(axis=0),
                                           rtol=1e-12, atol=1e-13)
                assert abs(lse[b, h, i] - (s + math.log(len(vis)))) < 1e-12


def test_causal_first_row_is_first_value_row(oracle):
    inp = fixed_inputs(B=2, H=2, H_k=1, Sq=10, Sk=10, D=16, mask="causal", seed=12)
    o, lse = oracle_on(oracle, inp)
    Q, K, V = exact(inp.q), exact(inp.k), exact(inp.v)
    o = o.reshape(2, 2, 10, 16)
    lse = lse.reshape(2, 2, 10)
    for b in range(2):
        for h in range(2):
            assert np.array_equal(o[b, h, 0], V[b, 0, 0])
            s00 = inp.w.softmax_scale * float(np.dot(Q[b, 0, h], K[b, 0, 0]))
            assert abs(lse[b, h, 0] - s00) < 1e-13


def test_causal_qend_rows_without_keys_and_single_key_row(oracle):
    """q-end with more queries than keys: rows i < Sq-Sk see nothing (O=0,
    LSE=-inf), row Sq-Sk sees exactly key 0."""
    Sq, Sk = 9, 4
    inp = fixed_inputs(B=1, H=1, H_k=1, Sq=Sq, Sk=Sk, D=8, mask="causal", causal_type="qend",
                       seed=13)
    o, lse = oracle_on(oracle, inp)
    V = exact(inp.v)
    for i in range(Sq - Sk):
        assert np.all(o[i] == 0) and lse[i] == -np.inf
    assert np.array_equal(o[Sq - Sk], V[0, 0, 0])


@pytest.mark.parametrize("Sq,Sk", [(5, 11), (11, 5)])
def test_one_dominant_key_closed_form(oracle, Sq, Sk):
    """Q rows c*e_0 and one key e_0 (all other keys 0): the scores are c*scale
    for that key and 0 elsewhere, so O and LSE have closed forms.  The chosen key
    differs per batch and kv head, which exposes index or operand mix-ups."""
    B, H, H_k, D = 2, 4, 2, 16
    inp = fixed_inputs(B=B, H=H, H_k=H_k, Sq=Sq, Sk=Sk, D=D, seed=14)
    c = 8.0
    inp.q.zero_()
    inp.q[..., 0] = c
    inp.k.zero_()
    star = {}
    for b in range(B):
        for g in range(H_k):
            j = (3 * b + 2 * g + 1) % Sk
            star[b, g] = j
            inp.k[b, j, g, 0] = 1.0
    o, lse = oracle_on(oracle, inp)
    o = o.reshape(B, H, Sq, D)
    lse = lse.reshape(B, H, Sq)
    V = exact(inp.v)
    sc = inp.w.softmax_scale
    e = math.exp(c * sc)
    for b in range(B):
        for h in range(H):
            g = h // (H // H_k)
            j = star[b, g]
            others = [x for x in range(Sk) if x != j]
            want = (e * V[b, j, g] + V[b, others, g].sum(axis=0)) / (e + Sk - 1)
            for i in range(Sq):
                np.testing.assert_allclose(o[b, h, i], want, rtol=1e-12, atol=1e-13)
                assert abs(lse[b, h, i] - math.log(e + Sk - 1)) < 1e-12


# ----------------------------------------------------------------------------
# attention: invariants
# ----------------------------------------------------------------------------

def test_key_permutation_invariance(oracle):
    inp = fixed_inputs(B=2, H=2, H_k=2, Sq=7, Sk=19, D=16, seed=15)
    o1, l1 = oracle_on(oracle, inp)
    perm = torch.randperm(19, generator=torch.Generator().manual_seed(3))
    inp.k[:] = inp.k[:, perm].clone()
    inp.v[:] = inp.v[:, perm].clone()
    o2, l2 = oracle_on(oracle, inp)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("H,H_k", [(4, 2), (6, 1), (8, 4)])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_gqa_equals_mha_with_repeated_kv_heads(oracle, H, H_k, mask):
    inp = fixed_inputs(B=2, H=H, H_k=H_k, Sq=9, Sk=9, D=8, mask=mask, seed=16)
    o1, l1 = oracle_on(oracle, inp)
    rep = H // H_k
    w2 = wl.Workload("t", dtype="bf16", B=2, H=H, H_k=H, Sq=9, Sk=9, D=8, mask=mask)
    inp2 = wl.Inputs(w2, inp.q, inp.k.repeat_interleave(rep, dim=2).contiguous(),
                     inp.v.repeat_interleave(rep, dim=2).contiguous())
    o2, l2 = oracle_on(oracle, inp2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("mask,ct", [("none", "qbegin"), ("causal", "qbegin"), ("causal", "qend")])
def test_varlen_equals_per_sequence_calls(oracle, mask, ct):
    lq, lk = [5, 0, 9, 3, 4], [7, 4, 0, 3, 2]
    inp = varlen_inputs(lq, lk, H=4, H_k=2, D=8, mask=mask, causal_type=ct, seed=17)
    o, lse = oracle_on(oracle, inp)
    T = inp.total_length
    o = o.reshape(4, T, 8)
    lse = lse.reshape(4, T)
    cq, ck = inp.cu_seqlens_q.tolist(), inp.cu_seqlens_k.tolist()
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        w1 = wl.Workload("t", dtype="bf16", B=1, H=4, H_k=2, Sq=lq[b], Sk=lk[b], D=8, mask=mask,
                         causal_type=ct)
        one = wl.Inputs(w1, inp.q[cq[b]:cq[b + 1]].unsqueeze(0).contiguous(),
                        inp.k[ck[b]:ck[b + 1]].unsqueeze(0).contiguous(),
                        inp.v[ck[b]:ck[b + 1]].unsqueeze(0).contiguous())
        o1, l1 = oracle_on(oracle, one)
        o1 = o1.reshape(4, lq[b], 8)
        l1 = l1.reshape(4, lq[b])
        assert np.array_equal(o[:, cq[b]:cq[b + 1]], o1)
        assert np.array_equal(lse[:, cq[b]:cq[b + 1]], l1)
        if lk[b] == 0:                    # a sequence with no keys
            assert np.all(o1 == 0) and np.all(l1 == -np.inf)
    # rows past the last sequence belong to nobody
    if cq[-1] < T:
        assert np.all(np.isnan(lse[:, cq[-1]:]))


def test_qbegin_equals_qend_for_square_problems(oracle):
    inp = fixed_inputs(B=1, H=2, H_k=1, Sq=11, Sk=11, D=8, mask="causal", seed=18)
    a = oracle_on(oracle, inp, causal_type="qbegin")
    b = oracle_on(oracle, inp, causal_type="qend")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_residual_equals_none(oracle):
    inp = fixed_inputs(B=1, H=2, H_k=2, Sq=5, Sk=13, D=8, seed=19)
    a = oracle_on(oracle, inp, mask="none")
    b = oracle_on(oracle, inp, mask="residual")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_out_scale_is_linear_and_leaves_lse(oracle):
    inp = fixed_inputs(B=1, H=2, H_k=2, Sq=6, Sk=9, D=8, mask="causal", seed=20)
    o1, l1 = oracle_on(oracle, inp, out_scale=1.0)
    o2, l2 = oracle_on(oracle, inp, out_scale=2.0)
    assert np.array_equal(2.0 * o1, o2) and np.array_equal(l1, l2)


def test_row_selection_matches_full(oracle):
    inp = fixed_inputs(B=2, H=3, H_k=1, Sq=17, Sk=23, D=8, mask="causal", causal_type="qend",
                       seed=21)
    o, lse = oracle_on(oracle, inp)
    rows = np.array([0, 5, 16, 17, 40, 101, 2 * 3 * 17 - 1], dtype=np.int64)
    o2, l2 = oracle_on(oracle, inp, rows=rows)
    assert np.array_equal(o[rows], o2) and np.array_equal(lse[rows], l2)


# ----------------------------------------------------------------------------
# brute force on tiny inputs: a different route (no max shift, exact sums)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mask,ct,Sq,Sk", [("none", "qbegin", 3, 5), ("causal", "qbegin", 5, 5),
                                           ("causal", "qend", 3, 6), ("causal", "qend", 6, 3),
                                           ("causal", "qbegin", 6, 3), ("residual", "qbegin", 4, 7)])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
def test_brute_force_tiny(oracle, mask, ct, Sq, Sk, dtype):
    B, H, H_k, D = 2, 2, 1, 4
    inp = fixed_inputs(dtype=dtype, B=B, H=H, H_k=H_k, Sq=Sq, Sk=Sk, D=D, mask=mask,
                       causal_type=ct, seed=22)
    o, lse = oracle_on(oracle, inp)
    o = o.reshape(B, H, Sq, D)
    lse = lse.reshape(B, H, Sq)
    Q, K, V = exact(inp.q).tolist(), exact(inp.k).tolist(), exact(inp.v).tolist()
    sc = inp.w.softmax_scale
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                vis = _allowed(mask, ct, i, Sq, Sk)
                if not vis:
                    assert all(x == 0 for x in o[b, h, i]) and lse[b, h, i] == -math.inf
                    continue
                e = {j: math.exp(sc * math.fsum(Q[b][i][h][d] * K[b][j][0][d] for d in range(D)))
                     for j in vis}
                z = math.fsum(e.values())
                for d in range(D):
                    want = math.fsum(e[j] / z * V[b][j][0][d] for j in vis)
                    assert abs(o[b, h, i, d] - want) <= 1e-12 * (1 + abs(want))
                assert abs(lse[b, h, i] - math.log(z)) <= 1e-12 * (1 + abs(math.log(z)))


def test_oracle_rejects_inconsistent_arguments(oracle):
    inp = fixed_inputs()
    with pytest.raises(ValueError):
        oracle.fmha_fwd(wl.bits(inp.q), wl.bits(inp.k), wl.bits(inp.v), 1, 1, 3, 2, 16, 16, 8,
                        0.3)                                  # H % H_k != 0
