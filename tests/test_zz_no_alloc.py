"""The allocation-free split-KV entry point, through the C ABI.

fmha_fwd_splitkv_noalloc serves callers that must not allocate device memory
while they run (a process that reserved its memory up front, a plug-in whose
host framework owns all allocations); it keeps its scratch in a fixed array
inside the library.  These tests check it against fmha_fwd_splitkv with a
caller workspace on two calls in a row -- different problem sizes, so scratch
left over from the first call would show in the second -- and that it rejects
a problem too big for the array.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import TOL_LSE, TOL_O, half_ulp
from tests.helpers import fixed_inputs, oracle_on, varlen_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


def _problem(fm, **kw):
    inp = fixed_inputs(dtype="bf16", D=128, **kw)
    w = inp.w
    dev_in = (inp.q.cuda(), inp.k.cuda(), inp.v.cuda())
    outs = []
    for _ in range(2):                       # one set for each entry point
        outs.append((torch.full(inp.q.shape, float("nan"), dtype=inp.q.dtype, device="cuda"),
                     torch.full((w.B, w.H, w.Sq), float("nan"), dtype=torch.float32, device="cuda")))
    return inp, dev_in, outs


def _call_pair(fm, inp, dev_in, outs, splits):
    w = inp.w
    scalars = (w.B, w.H, w.H_k, w.Sq, w.Sk, w.D, w.softmax_scale, w.out_scale,
               {"none": 0, "causal": 2}[w.mask], {"qbegin": 0, "qend": 1}[w.causal_type])
    (o_ref, l_ref), (o_na, l_na) = outs
    nbytes = fm.fmha_fwd_splitkv_workspace_size(w.B, w.H, w.Sq, w.D, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc = fm.fmha_fwd_splitkv(*dev_in, o_ref, l_ref, *scalars, num_splits=splits, workspace=ws)
    assert rc == 0, fm.status_string(rc)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    rc = fm.fmha_fwd_splitkv_noalloc(*dev_in, o_na, l_na, *scalars, num_splits=splits)
    assert rc == 0, fm.status_string(rc)
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    return free_before, torch.cuda.mem_get_info()[0]


def _check(inp, outs):
    (o_ref, l_ref), (o_na, l_na) = outs
    assert not torch.isnan(o_na).any() and not torch.isnan(l_na).any()
    assert (o_na.float() - o_ref.float()).abs().max().item() <= TOL_O[inp.w.dtype]
    fin = torch.isfinite(l_ref)
    assert torch.equal(torch.isfinite(l_na), fin)
    assert (l_na[fin] - l_ref[fin]).abs().max().item() <= TOL_LSE


def test_noalloc_matches_workspace_entry_on_two_calls(fm):
    # first call: causal q-end, 4 key ranges
    a = _problem(fm, B=1, H=4, H_k=2, Sq=300, Sk=2000, mask="causal", causal_type="qend", seed=41)
    _call_pair(fm, *a, splits=4)
    _check(a[0], a[2])
    # second call, smaller and with a different split count: stale partial
    # results of the first call are still in the shared array
    b = _problem(fm, B=2, H=2, H_k=1, Sq=200, Sk=1500, mask="none", seed=42)
    free_before, free_after = _call_pair(fm, *b, splits=3)
    _check(b[0], b[2])
    assert free_after >= free_before          # the call reserved no device memory


def test_noalloc_at_the_size_limit(fm):
    # B=1, H=2, D=128, 4 splits: Sq = 8128 needs all but 2 KB of the 32 MiB
    # array, so every partial result lands at the far end of it
    a = _problem(fm, B=1, H=2, H_k=2, Sq=8128, Sk=700, mask="causal", causal_type="qend", seed=43)
    assert fm.fmha_fwd_splitkv_workspace_size(1, 2, 8128, 128, 4) <= 32 << 20
    _call_pair(fm, *a, splits=4)
    _check(a[0], a[2])


def test_noalloc_varlen_against_the_oracle(fm, oracle):
    inp = varlen_inputs([300, 0, 517, 129], [700, 40, 517, 1000], dtype="bf16", H=4, H_k=2, D=128,
                        mask="causal", causal_type="qend", seed=44)
    w, T = inp.w, inp.total_length
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    cq, ck = inp.cu_seqlens_q.cuda(), inp.cu_seqlens_k.cuda()
    o = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full((w.H, T), float("nan"), dtype=torch.float32, device="cuda")
    rc = fm.fmha_fwd_splitkv_noalloc(q, k, v, o, lse, len(inp.seqlens_q), w.H, w.H_k, 0, 0, w.D,
                                     w.softmax_scale, 1.0, 2, 1, cq, ck, inp.max_len, T, num_splits=3)
    assert rc == 0, fm.status_string(rc)
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    end = int(inp.cu_seqlens_q[-1])
    rows = np.array([h * T + t for h in range(w.H) for t in range(end)], dtype=np.int64)
    o_ref, lse_ref = oracle_on(oracle, inp, rows=rows)
    got = o[:end].permute(1, 0, 2).reshape(-1, w.D).double().cpu().numpy()
    assert (np.abs(got - o_ref) <= TOL_O["bf16"] + half_ulp("bf16", o_ref)).all()
    got_lse = lse[:, :end].reshape(-1).double().cpu().numpy()
    masked = np.isneginf(lse_ref)
    assert np.isneginf(got_lse[masked]).all() and (got[masked] == 0).all()
    assert (np.abs(got_lse[~masked] - lse_ref[~masked]) <= TOL_LSE).all()


def test_noalloc_rejects_problems_larger_than_its_scratch(fm):
    B, H, Sq, D, splits = 1, 32, 8192, 128, 4
    need = fm.fmha_fwd_splitkv_workspace_size(B, H, Sq, D, splits)
    assert need > 32 << 20
    q = torch.zeros((B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    rc = fm.fmha_fwd_splitkv_noalloc(q, q, q, o, None, B, H, H, Sq, Sq, D, D ** -0.5, 1.0, 0, 0,
                                     num_splits=splits)
    assert rc == fm.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())             # nothing was launched
