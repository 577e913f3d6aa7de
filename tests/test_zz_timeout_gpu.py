"""The failure path of the forward, generation and backward kernels on the
GPU, without a fault: with the bounded waits limited to 1 ms, the producer of
every CTA first waits for a flag that nothing sets (fmha_set_test_gate), so
that wait runs out.  The call must report FMHA_ERR_TIMEOUT through fmha_device_status,
stop every role, free its tensor memory and leave the context usable: with
the gate off and the default limit back, the same call then matches the
oracle."""
import numpy as np
import pytest
import torch

from head_attention_forward_02_gb300 import workloads as wl
from tests.gpu_util import Run, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("e4m3", 128)])
def test_expired_wait_is_reported_and_the_context_stays_usable(fm, oracle, dtype, D):
    w = wl.Workload(f"timeout_{dtype}_d{D}", dtype=dtype, B=2, H=4, H_k=4, Sq=2048, Sk=2048, D=D,
                    mask="causal", seed=3)
    inp = wl.generate(w)
    assert fm.device_status(reset=True) == 0
    assert fm.set_wait_limit_ns(1_000_000) == 0
    assert fm.set_test_gate(True) == 0
    try:
        expired = Run(fm, inp)                 # reads and resets the device status
    finally:
        assert fm.set_test_gate(False) == 0
        assert fm.set_wait_limit_ns(0) == 0
    assert expired.status == fm.ERR_TIMEOUT
    again = Run(fm, inp)
    assert again.status == 0
    assert again.guards_intact()
    # rows of every (b, h), spread over the sequence
    rows = np.concatenate([bh * w.Sq + np.arange(0, w.Sq, 61) for bh in range(w.B * w.H)])
    compare(again, oracle, rows)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_generation_expired_wait_is_reported_and_the_context_stays_usable(fm, dtype):
    """The same for fmha_gen_fwd: its attention CTAs stop, the merge runs on
    undefined partials, the status reads FMHA_ERR_TIMEOUT, and the next call
    (gate off, default limit) matches the oracle."""
    from tests import test_gen_gpu as tg
    c = tg.make(dtype, 8, 32, 8, 8, 2048, [2047, 1000, 1, 0, 517, 1999, 64, 1500], False, seed=13,
                nan_tail=False)
    assert fm.device_status(reset=True) == 0
    assert fm.set_wait_limit_ns(1_000_000) == 0
    assert fm.set_test_gate(True) == 0
    try:
        _, _, _, _, status = tg.run(fm, c)
    finally:
        assert fm.set_test_gate(False) == 0
        assert fm.set_wait_limit_ns(0) == 0
    assert status == fm.ERR_TIMEOUT
    o, lse, _, _, status = tg.run(fm, c)
    assert status == 0
    tg.check(c, o, lse)


def test_backward_expired_wait_is_reported_and_the_context_stays_usable(fm):
    """The same for fmha_bwd: with the gate on, its dQ and dK/dV CTAs stop
    before any copy and the status reads FMHA_ERR_TIMEOUT; with the gate off
    the next call's gradients match the oracle."""
    from tests import test_bwd_gpu as tb
    g = torch.Generator().manual_seed(17)
    q, k, v, do = (torch.randn(1, 512, 4, 128, generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fm.fwd(qd, kd, vd, mask="causal")
    torch.cuda.synchronize()
    assert fm.device_status(reset=True) == 0
    assert fm.set_wait_limit_ns(1_000_000) == 0
    assert fm.set_test_gate(True) == 0
    try:
        fm.bwd(qd, kd, vd, o, dod, lse, mask="causal")
        torch.cuda.synchronize()
        status = fm.device_status(reset=True)
    finally:
        assert fm.set_test_gate(False) == 0
        assert fm.set_wait_limit_ns(0) == 0
    assert status == fm.ERR_TIMEOUT
    tb.run_case(fm, "bf16", 1, 4, 512, 512, 128, "causal", "qbegin", seed=17)
