"""Pins of the generation-phase oracle (one new query token against a K/V cache).

Each test fixes a value the definition determines independently of the oracle's
loop: a closed form, an invariance of the definition, or agreement with the
prefill oracle (pinned on its own in test_oracle_pins.py) on the same keys.
Source: "CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 生成阶段.
"""
import math

import numpy as np
import pytest

import oracle

BF16, F16, E4M3 = oracle.BF16, oracle.F16, oracle.E4M3


def enc(dtype, x):
    return oracle.encode(dtype, np.asarray(x, dtype=np.float64))


def dec(dtype, bits):
    return oracle.decode(dtype, bits)


def problem(seed, B=3, H=4, H_k=2, D=128, B_cache=4, S_max=40, dtype=BF16):
    rng = np.random.default_rng(seed)
    return dict(
        q=enc(dtype, rng.standard_normal((B, H, D))),
        kc=enc(dtype, rng.standard_normal((B_cache, S_max, H_k, D))),
        vc=enc(dtype, rng.standard_normal((B_cache, S_max, H_k, D))),
        kn=enc(dtype, rng.standard_normal((B, H_k, D))),
        vn=enc(dtype, rng.standard_normal((B, H_k, D))),
        B=B, H=H, H_k=H_k, D=D, B_cache=B_cache, S_max=S_max, dtype=dtype)


def run(p, seqlen, batch_idx=None, insert=True, scale=None, out_scale=1.0, **over):
    a = dict(p)
    a.update(over)
    scale = a["D"] ** -0.5 if scale is None else scale
    return oracle.gen_fwd(a["q"], a["kc"], a["vc"], a["kn"] if insert else None,
                          a["vn"] if insert else None, a["dtype"], a["B"], a["H"], a["H_k"],
                          a["D"], a["B_cache"], a["S_max"], np.asarray(seqlen, np.int32),
                          None if batch_idx is None else np.asarray(batch_idx, np.int32),
                          scale, out_scale)


@pytest.mark.parametrize("dtype", [BF16, E4M3])
def test_single_new_key_returns_its_value_exactly(dtype):
    p = problem(1, dtype=dtype)
    o, lse = run(p, [0, 0, 0])
    vn, kn, q = dec(dtype, p["vn"]), dec(dtype, p["kn"]), dec(dtype, p["q"])
    for b in range(3):
        for h in range(4):
            g = h // 2
            assert np.array_equal(o[b * 4 + h], vn[b, g])
            s = (p["D"] ** -0.5) * float(np.dot(q[b, h], kn[b, g]))
            assert lse[b * 4 + h] == pytest.approx(s, abs=1e-12)


def test_cache_only_without_tokens_gives_zero_and_minus_infinity():
    o, lse = run(problem(2), [0, 3, 0], insert=False)
    for r in list(range(0, 4)) + list(range(8, 12)):
        assert np.all(o[r] == 0) and lse[r] == -math.inf
    assert np.all(np.isfinite(lse[4:8]))


def test_equal_keys_give_the_mean_of_the_values():
    p = problem(3)
    key = enc(BF16, np.random.default_rng(9).standard_normal(p["D"]))
    kc = np.broadcast_to(key, p["kc"].shape).copy()
    kn = np.broadcast_to(key, p["kn"].shape).copy()
    seqlen = [5, 17, 1]
    o, lse = run(p, seqlen, kc=kc, kn=kn)
    vc, vn, q = dec(BF16, p["vc"]), dec(BF16, p["vn"]), dec(BF16, p["q"])
    kd = dec(BF16, key)
    for b, L in enumerate(seqlen):
        for h in range(4):
            g = h // 2
            vals = np.concatenate([vc[b, :L, g], vn[b, g][None]], axis=0)
            assert np.allclose(o[b * 4 + h], vals.mean(axis=0), atol=1e-12)
            s = (p["D"] ** -0.5) * float(np.dot(q[b, h], kd))
            assert lse[b * 4 + h] == pytest.approx(s + math.log(L + 1), abs=1e-12)


def test_insert_equals_cache_only_with_the_new_row_appended():
    p = problem(4)
    seqlen = [7, 0, 12]
    o_ins, lse_ins = run(p, seqlen)
    kc, vc = p["kc"].copy(), p["vc"].copy()
    for b, L in enumerate(seqlen):
        kc[b, L] = p["kn"][b]
        vc[b, L] = p["vn"][b]
    o_co, lse_co = run(p, [L + 1 for L in seqlen], insert=False, kc=kc, vc=vc)
    assert np.allclose(o_ins, o_co, atol=1e-13) and np.allclose(lse_ins, lse_co, atol=1e-13)


def test_batch_remap_reads_the_mapped_entry():
    p = problem(5)
    seqlen = [9, 4, 30]
    o_ref, lse_ref = run(p, seqlen, batch_idx=[0, 1, 2])
    perm = np.array([3, 0, 2, 1])            # entry e of the new cache holds old entry perm[e]
    kc, vc = p["kc"][perm], p["vc"][perm]
    where = [int(np.where(perm == b)[0][0]) for b in range(3)]
    o, lse = run(p, seqlen, batch_idx=where, kc=kc, vc=vc)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)
    # and a wrong map gives a different answer (the map is not ignored)
    o_bad, _ = run(p, seqlen, batch_idx=[0, 1, 2], kc=kc, vc=vc)
    assert not np.allclose(o_bad, o_ref)


@pytest.mark.parametrize("dtype", [BF16, E4M3])
def test_gqa_equals_mha_with_repeated_kv_heads(dtype):
    p = problem(6, H=8, H_k=2, dtype=dtype)
    seqlen = [3, 11, 25]
    o, lse = run(p, seqlen)
    rep = lambda x: np.repeat(x, 4, axis=-2)
    o2, lse2 = run(p, seqlen, H_k=8, kc=rep(p["kc"]), vc=rep(p["vc"]), kn=rep(p["kn"]), vn=rep(p["vn"]))
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("dtype", [F16, E4M3])
def test_matches_the_prefill_oracle_on_the_same_keys(dtype):
    p = problem(7, dtype=dtype)
    seqlen, bidx = [6, 0, 33], [2, 3, 0]
    o, lse = run(p, seqlen, batch_idx=bidx, out_scale=0.75)
    for b, (L, c) in enumerate(zip(seqlen, bidx)):
        k = np.concatenate([p["kc"][c, :L], p["kn"][b][None]], axis=0)[None]   # [1, L+1, H_k, D]
        v = np.concatenate([p["vc"][c, :L], p["vn"][b][None]], axis=0)[None]
        q = p["q"][b][None, None]                                            # [1, 1, H, D]
        o_p, lse_p = oracle.fmha_fwd(q, k, v, dtype, 1, 4, 2, 1, L + 1, 128, 128 ** -0.5, 0.75)
        assert np.allclose(o[b * 4:(b + 1) * 4], o_p, atol=1e-12)
        assert np.allclose(lse[b * 4:(b + 1) * 4], lse_p, atol=1e-12)


def test_out_scale_is_linear_and_leaves_lse_alone():
    p = problem(8)
    o1, l1 = run(p, [4, 9, 2])
    o2, l2 = run(p, [4, 9, 2], out_scale=2.0)
    assert np.allclose(o2, 2 * o1, atol=1e-13) and np.array_equal(l1, l2)


@pytest.mark.parametrize("seqlen,bidx,insert", [
    ([40, 0, 0], None, True),        # no room for the new token
    ([41, 0, 0], None, False),       # more tokens than the cache holds
    ([-1, 0, 0], None, False),
    ([1, 1, 1], [0, 4, 1], True),    # entry index out of range
])
def test_rejects_inconsistent_arguments(seqlen, bidx, insert):
    with pytest.raises(ValueError):
        run(problem(9), seqlen, batch_idx=bidx, insert=insert)
