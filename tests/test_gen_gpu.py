"""Generation-phase attention (fmha_gen_fwd) against the oracle, on the GPU.

Cases cover fp16, bf16 and e4m3, insert and cache-only modes, batch remapping,
head groups of 1 to 32, work units of one kv head (odd H_k, or query groups
wider than 16) and of two adjacent kv heads (64-key tiles), lengths at tile
and chunk edges (the key range is cut into chunks of whole tiles), an empty
cache, NaN-filled rows past every length, the cache rows the call writes, and
a length outside the cache (reported, not a fault).  e4m3 inputs are compared
with the oracle on their decoded values.
"""
import numpy as np
import pytest
import torch

import oracle
from head_attention_forward_02_gb300 import workloads as wl
from tests.gpu_util import TOL_LSE, TOL_O, half_ulp

pytestmark = pytest.mark.gpu

DT = {"bf16": (torch.bfloat16, oracle.BF16), "f16": (torch.float16, oracle.F16),
      "e4m3": (torch.float8_e4m3fn, oracle.E4M3)}
MEAN_TOL = {"bf16": 1e-3, "f16": 1e-3, "e4m3": 1e-2}


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


def make(dtype, B, H, H_k, B_cache, S_max, seqlen, insert, seed, batch_idx=None, nan_tail=True):
    tdt, _ = DT[dtype]
    g = torch.Generator().manual_seed(seed)
    rnd = lambda *s: torch.randn(*s, generator=g).to(tdt)
    kc, vc = rnd(B_cache, S_max, H_k, 128), rnd(B_cache, S_max, H_k, 128)
    if nan_tail:
        # rows past each sequence's keys hold NaN: they must never reach O
        for b, L in enumerate(seqlen):
            e = b if batch_idx is None else batch_idx[b]
            kc[e, L:] = float("nan")
            vc[e, L:] = float("nan")
    return dict(q=rnd(B, H, 128), kc=kc, vc=vc, kn=rnd(B, H_k, 128) if insert else None,
                vn=rnd(B, H_k, 128) if insert else None, seqlen=torch.tensor(seqlen, dtype=torch.int32),
                bidx=None if batch_idx is None else torch.tensor(batch_idx, dtype=torch.int32),
                B=B, H=H, H_k=H_k, B_cache=B_cache, S_max=S_max, dtype=dtype)


def bits(t):
    if t is None:
        return None
    return t.view(torch.uint8 if t.element_size() == 1 else torch.uint16).numpy()


def run(fm, c, out_scale=1.0):
    dev = torch.device("cuda")
    kc, vc = c["kc"].to(dev), c["vc"].to(dev)
    o, lse = fm.gen_fwd(c["q"].to(dev), kc, vc, c["seqlen"].to(dev),
                        k_new=None if c["kn"] is None else c["kn"].to(dev),
                        v_new=None if c["vn"] is None else c["vn"].to(dev),
                        batch_idx=None if c["bidx"] is None else c["bidx"].to(dev), out_scale=out_scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu(), kc.cpu(), vc.cpu(), fm.device_status(reset=True)


def reference(c, out_scale=1.0):
    """The oracle reads the cache as it was before the call."""
    _, odt = DT[c["dtype"]]
    return oracle.gen_fwd(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), bits(c["kn"]), bits(c["vn"]), odt,
                          c["B"], c["H"], c["H_k"], 128, c["B_cache"], c["S_max"], c["seqlen"].numpy(),
                          None if c["bidx"] is None else c["bidx"].numpy(), 128 ** -0.5, out_scale)


def check(c, o, lse, out_scale=1.0, extra=None):
    """O within tol + half an output ulp (+ extra), mean error within the mean
    tolerance plus the mean half ulp; LSE within TOL_LSE; empty rows 0 / -inf."""
    o_ref, lse_ref = reference(c, out_scale)
    got = o.float().numpy().reshape(-1, 128).astype(np.float64)
    assert not np.isnan(got).any(), "NaN in O"
    err = np.abs(got - o_ref)
    hu = half_ulp(c["dtype"], o_ref)
    bound = TOL_O[c["dtype"]] + hu + (0.0 if extra is None else extra)
    assert (err <= bound).all(), f"O mismatch: worst {err.max():.4g} at row {np.argwhere(err > bound)[0][0]}"
    assert err.mean() <= MEAN_TOL[c["dtype"]] + hu.mean() + (0.0 if extra is None else extra.mean()), err.mean()
    l = lse.numpy().reshape(-1).astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(l[empty])) and np.all(got[empty] == 0)
    assert np.abs(l[~empty] - lse_ref[~empty]).max(initial=0.0) <= TOL_LSE


def check_cache(c, kc, vc):
    """Insert mode writes exactly row L of each sequence's entry (kv heads of
    that sequence); everything else is unchanged."""
    kc_ref, vc_ref = c["kc"].clone(), c["vc"].clone()
    if c["kn"] is not None:
        for b, L in enumerate(c["seqlen"].tolist()):
            e = b if c["bidx"] is None else int(c["bidx"][b])
            kc_ref[e, L] = c["kn"][b]
            vc_ref[e, L] = c["vn"][b]
    assert np.array_equal(bits(kc), bits(kc_ref))
    assert np.array_equal(bits(vc), bits(vc_ref))


CASES = [
    # dtype, B, H, H_k, B_cache, S_max, seqlen, insert, batch_idx
    ("bf16", 4, 8, 2, 5, 1000, [0, 1, 517, 998], True, [3, 1, 0, 4]),
    ("f16", 4, 32, 1, 4, 300, [128, 129, 255, 1], False, None),
    ("bf16", 3, 16, 16, 3, 4096, [895, 1791, 4095], True, None),
    ("f16", 5, 4, 4, 6, 700, [127, 0, 640, 2, 383], True, [5, 0, 2, 1, 3]),
    ("bf16", 2, 12, 4, 2, 2048, [2047, 1024], False, [1, 0]),
    ("bf16", 6, 8, 8, 6, 513, [0, 0, 0, 512, 0, 0], False, None),      # mostly empty caches
    ("bf16", 3, 6, 3, 3, 700, [64, 63, 639], True, [2, 0, 1]),          # odd H_k: one kv head per unit
    ("f16", 2, 40, 2, 2, 400, [65, 399], True, None),                   # G = 20: one kv head per unit
    ("e4m3", 2, 32, 2, 2, 400, [64, 398], True, None),                  # G = 16: two heads fill S^T
    ("bf16", 2, 48, 2, 2, 900, [300, 899], True, None),                 # G = 24: two column groups of 16
    ("e4m3", 3, 96, 3, 3, 500, [129, 0, 499], False, [1, 2, 0]),        # G = 32, odd H_k
    ("f16", 2, 6, 3, 2, 300, [1, 255], True, None),                     # G = 2, odd H_k
    ("e4m3", 4, 8, 2, 5, 1000, [0, 1, 517, 998], True, [3, 1, 0, 4]),
    ("e4m3", 4, 32, 1, 4, 300, [128, 129, 255, 1], False, None),
    ("e4m3", 3, 16, 16, 3, 4096, [895, 1791, 4095], True, None),
    ("e4m3", 5, 4, 4, 6, 700, [127, 0, 640, 2, 383], True, [5, 0, 2, 1, 3]),
    # e4m3 tiles of two 128-row blocks: 256 keys of one kv head, or 128 keys of two
    ("e4m3", 3, 6, 3, 3, 700, [64, 63, 639], True, [2, 0, 1]),          # G = 2, odd H_k
    ("e4m3", 2, 36, 3, 2, 1100, [257, 1023], True, None),               # G = 12, odd H_k
    ("e4m3", 3, 16, 2, 3, 900, [255, 256, 899], False, None),           # G = 8, two heads a unit
    ("e4m3", 2, 40, 2, 2, 400, [65, 399], True, None),                  # G = 20: one block, eight warps
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_b{c[1]}_h{c[2]}_hk{c[3]}_s{c[5]}_{'ins' if c[7] else 'co'}"
                                             for c in CASES])
def test_gen_matches_oracle(fm, case):
    dtype, B, H, H_k, B_cache, S_max, seqlen, insert, bidx = case
    c = make(dtype, B, H, H_k, B_cache, S_max, seqlen, insert, seed=B * 100 + H, batch_idx=bidx)
    o, lse, kc, vc, status = run(fm, c)
    assert status == 0
    check(c, o, lse)
    check_cache(c, kc, vc)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_gen_long_caches_and_out_scale(fm, dtype):
    rng = np.random.default_rng(11)
    seqlen = rng.integers(1, 8191, size=8).tolist()
    c = make(dtype, 8, 32, 8, 8, 8192, seqlen, True, seed=77, nan_tail=False)
    o, lse, kc, vc, status = run(fm, c, out_scale=0.5)
    assert status == 0
    check(c, o, lse, out_scale=0.5)
    check_cache(c, kc, vc)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_gen_one_long_sequence_among_many(fm, dtype):
    # 48 two-head units: one warp merges each row; the one long sequence's
    # rows meet over a hundred chunks (the merge's 32-chunk rounds and its
    # batches of eight); cache-only, four shared entries
    B = 48
    seqlen = [60000] + [1 + (37 * b) % 200 for b in range(1, B)]
    c = make(dtype, B, 8, 2, 4, 60000, seqlen, False, seed=91, batch_idx=[b % 4 for b in range(B)],
             nan_tail=False)
    o, lse, _, _, status = run(fm, c)
    assert status == 0
    check(c, o, lse)


def abs_v_bound(c):
    """2^-4 times the attention output of |V|: the most that rounding each
    weight to e4m3 (relative error 2^-4 in e4m3's normal range) can move O
    when the row sum adds the unrounded weights."""
    def absolute(t):   # clear the sign bit of every e4m3 code
        return None if t is None else (t.view(torch.uint8) & 0x7F).view(t.dtype)

    a = dict(c)
    a["vc"], a["vn"] = absolute(c["vc"]), absolute(c["vn"])
    o_abs, _ = reference(a)
    return 2.0 ** -4 * o_abs


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_gen_growing_scores_force_rescales(fm, dtype):
    # each sequence's keys lean more and more towards its first query head,
    # so that head's maximum keeps growing past the rescale threshold
    c = make(dtype, 2, 8, 2, 2, 1500, [1499, 900], False, seed=5, nan_tail=False)
    g = torch.Generator().manual_seed(6)
    ramp = torch.linspace(0.0, 3.0, 1500).view(1500, 1, 1)
    kc = 0.3 * torch.randn(2, 1500, 2, 128, generator=g)
    for b in range(2):
        qd = c["q"][b, 0].float()
        kc[b] += ramp * (4.0 * qd / qd.norm()).view(1, 1, 128)
    c["kc"] = kc.to(DT[dtype][0])
    o, lse, _, _, status = run(fm, c)
    assert status == 0
    check(c, o, lse, extra=abs_v_bound(c) if dtype == "e4m3" else None)


def test_gen_empty_batch(fm):
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 16, 2, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = fm.gen_fwd(q, kc, kc.clone(), torch.empty(0, dtype=torch.int32, device="cuda"))
    assert o.shape == (0, 8, 128)


def test_gen_length_outside_the_cache_is_reported(fm):
    # seqlen = S_max leaves no row for the new token: the kernel clamps,
    # inserts nothing and reports FMHA_ERR_INVALID_ARG
    c = make("bf16", 2, 4, 2, 2, 256, [256, 10], True, seed=3, nan_tail=False)
    c_ok = dict(c)
    _, _, kc, _, status = run(fm, c)
    assert status == fm.ERR_INVALID_ARG
    assert torch.equal(kc[0].view(torch.uint16), c_ok["kc"][0].view(torch.uint16))   # entry 0 untouched
    assert fm.device_status() == 0                                                      # reset by run()


@pytest.mark.parametrize("name", list(wl.GEN_CONFIGS))
def test_gen_full_size_configs(fm, name):
    """The benchmark's generation workloads at full size, through the same call
    the benchmark times: every output row against the oracle (which reads the
    caches as they were before the call) and the rows the call inserted."""
    w = wl.GEN_CONFIGS[name]
    inp = wl.generate_gen(w)
    dev = torch.device("cuda")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    o, lse = fm.gen_fwd(inp.q.to(dev), kc, vc, inp.seqlen.to(dev),
                        k_new=None if inp.k_new is None else inp.k_new.to(dev),
                        v_new=None if inp.v_new is None else inp.v_new.to(dev))
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    c = dict(q=inp.q, kc=inp.k_cache, vc=inp.v_cache, kn=inp.k_new, vn=inp.v_new, seqlen=inp.seqlen, bidx=None,
             B=w.B, H=w.H, H_k=w.H_k, B_cache=w.B, S_max=w.S_max, dtype=w.dtype)
    check(c, o.cpu(), lse.cpu())
    check_cache(c, kc.cpu(), vc.cpu())
