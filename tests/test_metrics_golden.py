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
