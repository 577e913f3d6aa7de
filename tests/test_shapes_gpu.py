"""GPU parity of the persistent forward kernel on many-unit problems.

Every instantiation of the tensor-core kernel (head dim 32 / 64 / 128, fp16 /
bf16 / e4m3, masked and unmasked) is run here on a problem with far more
(batch, head, 256-row query block) units than the GB300 has SMs, so each
persistent CTA takes many units in turn and reuses its Q slots, its K/V ring
phases and its accumulator barriers across units.  These are also the shapes
whose throughput the design record reports.  Heads 0 and H-1 of the first and
last batch are compared at tile-edge rows, plus a seeded sample of 1024 rows;
the oracle computes those rows one by one.  Guard bands around O and LSE must
be untouched.

Head dims and types: "FMHA for Blackwell: Forward" (head dims 32, 64 and 128;
fp8, fp16 and bf16 inputs).
"""
import pytest
import torch

from head_attention_forward_02_gb300 import workloads as wl
from tests.gpu_util import Run, compare, sample_rows
from tests.helpers import fixed_inputs, varlen_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


@pytest.mark.parametrize("name", list(wl.EXTRA_CONFIGS))
def test_benchmarked_shape(fm, oracle, name):
    """The extra workloads the benchmark times, at their full size and seed:
    bf16 causal D=64 (2048 units) and D=32 (1024), bf16 unmasked GQA S=8192
    (2048), bf16 causal S=16384 (2048), e4m3 causal GQA S=8192 (2048) and
    e4m3 causal D=64 (1024)."""
    w = wl.EXTRA_CONFIGS[name]
    inp = wl.generate(w)
    run = Run(fm, inp, "tc")
    assert run.status == 0
    assert run.guards_intact()
    stats = compare(run, oracle, sample_rows(inp, 1024, seed=w.seed))
    print(name, stats)


SHAPES = [
    # dtype, B, H, H_k, Sq, Sk, D, mask, causal_type     (units = B * H * ceil(Sq / 256))
    ("bf16", 2, 16, 4, 2048, 4096, 128, "causal", "qend"),        # 256, Sq < Sk
    ("bf16", 2, 16, 4, 2048, 4096, 64, "causal", "qend"),         # 256, Sq < Sk
    ("f16", 4, 16, 16, 2048, 2048, 128, "causal", "qbegin"),      # 512
    ("f16", 2, 16, 16, 4096, 4096, 64, "none", "qbegin"),         # 512
    ("f16", 2, 16, 8, 4096, 4096, 32, "causal", "qbegin"),        # 512
    ("e4m3", 2, 16, 16, 4096, 4096, 32, "none", "qbegin"),        # 512
    ("e4m3", 2, 16, 4, 3000, 5000, 64, "causal", "qend"),         # 384, ragged tails
]


def _id(c):
    return "-".join(str(x) for x in c)


@pytest.mark.parametrize("case", SHAPES, ids=[_id(c) for c in SHAPES])
def test_many_units(fm, oracle, case):
    dtype, B, H, H_k, Sq, Sk, D, mask, ct = case
    inp = fixed_inputs(dtype=dtype, B=B, H=H, H_k=H_k, Sq=Sq, Sk=Sk, D=D, mask=mask,
                       causal_type=ct, seed=sum(map(ord, _id(case))) % 997)
    run = Run(fm, inp, "tc")
    assert run.status == 0
    assert run.guards_intact()
    stats = compare(run, oracle, sample_rows(inp, 1024, seed=B * H + D))
    print(_id(case), stats)


VARLEN = [
    # dtype, H, H_k, D, number of sequences, length range, mask
    ("bf16", 16, 16, 64, 16, (256, 2048), "causal"),
    ("f16", 16, 4, 32, 24, (100, 3000), "causal"),
    ("e4m3", 16, 16, 128, 8, (256, 4096), "none"),
]


@pytest.mark.parametrize("case", VARLEN, ids=[_id(c) for c in VARLEN])
def test_many_units_varlen(fm, oracle, case):
    dtype, H, H_k, D, n, (lo, hi), mask = case
    g = torch.Generator().manual_seed(n * 31 + D)
    lens = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    inp = varlen_inputs(lens, lens, dtype=dtype, H=H, H_k=H_k, D=D, mask=mask, seed=n + D)
    run = Run(fm, inp, "tc")
    assert run.status == 0
    assert run.guards_intact()
    stats = compare(run, oracle, sample_rows(inp, 1024, seed=n))
    print(_id(case), stats)
