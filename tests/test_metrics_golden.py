"""The FLOP accounting reproduces the printed benchmark table of the sm120 page."""
import os

from head_attention_forward_02_gb300.metrics import algorithmic_bytes, attention_flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sm120_article_benchmark.txt")


def test_flops_reproduce_printed_tflops():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 5
    for s, t_ms, t_tf, f_ms, f_tf in rows:
        S = int(s)
        fl = attention_flops(1, 32, S, S, 128, causal=True)
        for ms, tf in ((t_ms, t_tf), (f_ms, f_tf)):
            assert abs(fl / (float(ms) * 1e-3) / 1e12 - float(tf)) < 0.006


def test_varlen_flops_sum_per_sequence():
    a = attention_flops(0, 16, 0, 0, 128, True, seqlens_q=[256, 1000], seqlens_k=[256, 1000])
    b = attention_flops(1, 16, 256, 256, 128, True) + attention_flops(1, 16, 1000, 1000, 128, True)
    assert a == b


def test_bytes_gqa_counts_kv_heads():
    assert algorithmic_bytes(2, 32, 8, 8192, 8192, 128, 2, 2) == \
        2 * 8192 * 32 * 128 * 2 * 2 + 2 * 2 * 8192 * 8 * 128 * 2 + 2 * 32 * 8192 * 4


def test_generation_bytes_and_flops_from_tensor_sizes():
    """gen_bytes / gen_flops against a direct count over a generated problem:
    the cached K/V rows each sequence attends, the new rows read and written,
    q, O and LSE; four flops (two products) per head dimension per key."""
    import torch

    from head_attention_forward_02_gb300 import workloads as wl
    from head_attention_forward_02_gb300.metrics import gen_bytes, gen_flops

    w = wl.GenWorkload("count", B=3, H=8, H_k=2, S_max=64, lengths="uniform", seed=5)
    inp = wl.generate_gen(w)
    lens = [int(x) for x in inp.seqlen]
    e = inp.q.element_size()
    row = inp.k_cache[0, 0].numel() * e                      # one cached token, all kv heads
    count = sum(2 * L * row for L in lens)                    # K and V rows attended
    count += 2 * 2 * inp.k_new.numel() * e                    # new K, V read and written
    count += 2 * inp.q.numel() * e + w.B * w.H * 4            # q in, O out, LSE out
    assert gen_bytes(w.B, w.H, w.H_k, lens, True, e) == count
    keys = [L + 1 for L in lens]                              # the new token is attended too
    flops = 0
    for k in keys:
        for _ in range(w.H):
            flops += k * (2 * 128 + 2 * 128)
    assert gen_flops(w.H, lens, True) == flops
    assert gen_flops(w.H, lens, False) == flops - len(lens) * w.H * 4 * 128


def test_backward_flops_convention():
    """bench.py's backward count: five products of 2*D flops per (query, key)
    pair; no mask counts every pair, a causal mask counts half of them (the
    pages' convention, S^2/2, rather than the S(S+1)/2 visible pairs)."""
    import bench

    B, H, S, D = 2, 3, 40, 64
    pairs = S * S
    assert bench.bwd_flops(B, H, S, D, False) == B * H * pairs * 5 * 2 * D
    visible = sum(1 for i in range(S) for j in range(S) if j <= i)
    assert visible == S * (S + 1) // 2
    assert bench.bwd_flops(B, H, S, D, True) == B * H * (S * S / 2) * 5 * 2 * D
