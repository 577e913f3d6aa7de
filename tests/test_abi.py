"""The C ABI without a GPU: symbols, argument validation, scheduler tile math."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fmha.h")


@pytest.fixture(scope="module")
def fm():
    from head_attention_forward_02_gb300 import build, fmha
    build.build()
    fmha.lib()
    return fmha


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(fmha_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fmha_fwd", "fmha_fwd_simt", "fmha_status_string", "fmha_device_status",
              "fmha_kv_tile_range"):
        assert n in names


def test_library_exports_every_declared_symbol(fm):
    L = fm.lib()
    for n in declared_functions():
        assert hasattr(L, n), n


def test_status_strings(fm):
    for code in (0, -1, -2, -3, -4):
        assert fm.status_string(code)
    assert fm.status_string(-99) == "unknown status"


P = 0x10000  # a fake, 16-byte aligned address: validation never dereferences


def call(fm, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, B=1, H=2, H_k=2, Sq=128, Sk=128, D=128,
             scale=0.1, out_scale=1.0, mask=0, causal_type=0, cu_seqlens_q=None,
             cu_seqlens_k=None, max_len=0, total_length=0, dtypes=(1, 1, 1, 1))
    a.update(kw)
    dq, dk, dv, do = a.pop("dtypes")
    L = fm.lib()
    return L.fmha_fwd(fm.fmha_tensor(a["q"], dq), fm.fmha_tensor(a["k"], dk),
                      fm.fmha_tensor(a["v"], dv), fm.fmha_tensor(a["o"], do), a["lse"],
                      a["B"], a["H"], a["H_k"], a["Sq"], a["Sk"], a["D"], a["scale"],
                      a["out_scale"], a["mask"], a["causal_type"], a["cu_seqlens_q"],
                      a["cu_seqlens_k"], a["max_len"], a["total_length"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), -1), (dict(D=256), -1), (dict(H=3, H_k=2), -1), (dict(H_k=0), -1),
    (dict(B=-1), -1), (dict(Sq=-5), -1), (dict(mask=3), -1), (dict(causal_type=2), -1),
    (dict(scale=float("nan")), -1), (dict(out_scale=float("inf")), -1),
    (dict(scale=0.0), -1), (dict(scale=-0.1), -1),
    (dict(cu_seqlens_q=P), -1),                                   # only one cu_seqlens
    (dict(cu_seqlens_q=P, cu_seqlens_k=P, total_length=-1, max_len=4), -1),
    (dict(cu_seqlens_q=P, cu_seqlens_k=P, total_length=10, max_len=0), -1),
    (dict(q=0), -1), (dict(o=0), -1),
    (dict(dtypes=(1, 0, 1, 1)), -2), (dict(dtypes=(2, 2, 2, 1)), -2), (dict(dtypes=(1, 1, 1, 7)), -1),
    (dict(q=P + 8), -2), (dict(v=P + 2), -2), (dict(lse=P + 2), -1),
])
def test_validation_rejects_before_any_launch(fm, kw, code):
    assert call(fm, **kw) == code


def test_empty_problems_succeed_without_a_device(fm):
    assert call(fm, B=0, q=0, k=0, v=0, o=0) == 0
    assert call(fm, Sq=0, q=0, k=0, v=0, o=0) == 0
    assert call(fm, cu_seqlens_q=P, cu_seqlens_k=P, total_length=0, max_len=0, B=3) == 0


def _brute(row0, rows, sq, sk, mask, ct, tn):
    last = min(row0 + rows, sq) - 1
    if last < row0 or sk <= 0:
        return 0, 0
    off = sk - sq if (mask == 2 and ct == 1) else 0

    def vis(i, j):
        return j < sk and (mask != 2 or j <= i + off)

    top = -1
    for i in range(row0, last + 1):
        for j in range(sk):
            if vis(i, j):
                top = max(top, j)
    n_tiles = 0 if top < 0 else top // tn + 1
    nu = 0
    while nu < n_tiles and all(vis(i, j) for i in range(row0, last + 1)
                               for j in range(nu * tn, (nu + 1) * tn)):
        nu += 1
    return n_tiles, nu


def test_kv_tile_range_matches_brute_force(fm):
    rng = np.random.default_rng(5)
    cases = [(0, 8, 9, 13, 2, 0, 4), (4, 8, 9, 5, 2, 1, 4), (0, 4, 3, 0, 0, 0, 4), (8, 8, 9, 20, 2, 1, 8)]
    for _ in range(400):
        tn = int(rng.choice([2, 4, 8]))
        sq, sk = int(rng.integers(0, 40)), int(rng.integers(0, 40))
        row0 = int(rng.integers(0, 40)) // tn * tn
        cases.append((row0, tn * int(rng.integers(1, 3)), sq, sk, int(rng.integers(0, 3)),
                      int(rng.integers(0, 2)), tn))
    for c in cases:
        assert fm.kv_tile_range(*c) == _brute(*c), c


def test_splitkv_workspace_size(fm):
    # fixed length: rows = B*Sq; LSE block rounded up to 256 bytes, then fp32 O
    n = fm.fmha_fwd_splitkv_workspace_size(2, 4, 100, 64, 3)
    lse = 3 * 200 * 4 * 4
    assert n == ((lse + 255) // 256) * 256 + 3 * 200 * 4 * 64 * 4
    # varlen: rows = total_length
    assert fm.fmha_fwd_splitkv_workspace_size(9, 2, 0, 128, 2, 77) == \
        ((2 * 77 * 2 * 4 + 255) // 256) * 256 + 2 * 77 * 2 * 128 * 4
    for bad in [(2, 4, 100, 96, 3), (2, 4, 100, 64, 0), (2, 4, 100, 64, 257), (2, 0, 100, 64, 1)]:
        assert fm.fmha_fwd_splitkv_workspace_size(*bad) == 0


def call_split(fm, ws=P, ws_bytes=1 << 30, splits=2, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, B=1, H=2, H_k=2, Sq=128, Sk=128, D=128, scale=0.1,
             out_scale=1.0, mask=0, causal_type=0)
    a.update(kw)
    t = [fm.fmha_tensor(a[x], 1) for x in "qkvo"]
    return fm.lib().fmha_fwd_splitkv(*t, a["lse"], a["B"], a["H"], a["H_k"], a["Sq"], a["Sk"], a["D"],
                                      a["scale"], a["out_scale"], a["mask"], a["causal_type"], None, None,
                                      0, 0, splits, ws, ws_bytes, None)


def test_splitkv_validation(fm):
    assert call_split(fm, splits=0) == -1
    assert call_split(fm, splits=257) == -1
    assert call_split(fm, ws=None) == -1
    assert call_split(fm, ws_bytes=100) == -1                  # too small
    assert call_split(fm, ws=P + 16) == -1                     # not 256-byte aligned
    assert call_split(fm, D=48) == -1
    assert call_split(fm, B=0, splits=3) == 0                  # nothing to do


def call_noalloc(fm, splits=2, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, B=1, H=2, H_k=2, Sq=128, Sk=128, D=128, scale=0.1,
             out_scale=1.0, mask=0, causal_type=0, cu_q=None, cu_k=None, max_len=0, total_length=0)
    a.update(kw)
    t = [fm.fmha_tensor(a[x], 1) for x in "qkvo"]
    return fm.lib().fmha_fwd_splitkv_noalloc(*t, a["lse"], a["B"], a["H"], a["H_k"], a["Sq"], a["Sk"],
                                              a["D"], a["scale"], a["out_scale"], a["mask"],
                                              a["causal_type"], a["cu_q"], a["cu_k"], a["max_len"],
                                              a["total_length"], splits, None)


# Every case below returns before the device is touched: the entry point
# checks its arguments as fmha_fwd_splitkv does, and only then its size limit.
@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 0), (dict(Sq=0), 0), (dict(B=0, q=None, k=None, v=None, o=None), 0),
    (dict(cu_q=P, cu_k=P, total_length=0, max_len=0, B=3), 0),      # empty varlen problem
    (dict(splits=0), -1), (dict(splits=257), -1), (dict(D=48), -1), (dict(H=3, H_k=2), -1),
    (dict(scale=0.0), -1), (dict(mask=5), -1), (dict(cu_q=P), -1), (dict(q=None), -1),
    (dict(q=P + 8), -2), (dict(lse=P + 2), -1),
    (dict(B=1, H=32, H_k=32, Sq=8192, Sk=8192, splits=4), -2),      # 34 MiB of scratch > 32 MiB
    (dict(B=1, H=33, H_k=2, Sq=8192, Sk=8192, splits=4), -1),       # too big and a bad head count
    (dict(cu_q=P, cu_k=P, total_length=1 << 20, max_len=4096, H=16, splits=2), -2),
])
def test_noalloc_validation_before_any_launch(fm, kw, code):
    assert call_noalloc(fm, **kw) == code


def test_noalloc_limit_is_the_split_kv_scratch_size(fm):
    # B=1, H=2, D=128, 4 splits: Sq = 8128 needs just under the 32 MiB array,
    # Sq = 8129 just over it (and is refused before any launch)
    limit = 32 << 20
    assert fm.fmha_fwd_splitkv_workspace_size(1, 2, 8128, 128, 4) <= limit
    assert fm.fmha_fwd_splitkv_workspace_size(1, 2, 8129, 128, 4) > limit
    assert call_noalloc(fm, H=2, H_k=2, Sq=8129, Sk=300, splits=4) == -2


def call_gen(fm, **kw):
    a = dict(q=P, kc=P, vc=P, kn=None, vn=None, o=P, lse=None, B=2, H=8, H_k=2, D=128, B_cache=2, S_max=64,
             seqlen=P, bidx=None, scale=0.1, out_scale=1.0, ws=P, ws_bytes=1 << 30, dtypes=(1, 1, 1, 1))
    a.update(kw)
    dq, dkc, dvc, do = a.pop("dtypes")
    t = fm.fmha_tensor
    return fm.lib().fmha_gen_fwd(t(a["q"], dq), t(a["kc"], dkc), t(a["vc"], dvc), t(a["kn"], dq),
                                 t(a["vn"], dq), t(a["o"], do), a["lse"], a["B"], a["H"], a["H_k"], a["D"],
                                 a["B_cache"], a["S_max"], a["seqlen"], a["bidx"], a["scale"],
                                 a["out_scale"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), -1), (dict(H=3, H_k=2), -1), (dict(H=64, H_k=1), -1), (dict(H_k=0), -1),
    (dict(B=-1), -1), (dict(scale=0.0), -1), (dict(scale=float("inf")), -1),
    (dict(out_scale=float("nan")), -1), (dict(kn=P), -1), (dict(vn=P), -1),
    (dict(S_max=0), -1), (dict(B_cache=0), -1), (dict(seqlen=None), -1), (dict(q=None), -1),
    (dict(o=None), -1), (dict(dtypes=(5, 5, 5, 5)), -2), (dict(dtypes=(1, 0, 1, 1)), -2),
    (dict(dtypes=(2, 2, 2, 1)), -2), (dict(dtypes=(2, 1, 1, 1)), -2),
    (dict(q=P + 8), -2), (dict(kc=P + 2), -2), (dict(lse=P + 2), -1),
])
def test_gen_validation_rejects_before_any_launch(fm, kw, code):
    assert call_gen(fm, **kw) == code


def test_gen_empty_batch_succeeds_without_a_device(fm):
    assert call_gen(fm, B=0, q=None, kc=None, vc=None, o=None, seqlen=None, ws=None) == 0


def test_gen_workspace_size_rejects_bad_sizes(fm):
    for bad in [(0, 8, 2, 128, 64), (2, 8, 3, 128, 64), (2, 8, 2, 64, 64), (2, 8, 2, 128, 0)]:
        assert fm.fmha_gen_workspace_size(*bad) == 0


@pytest.mark.parametrize("H,H_k,keys_per_tile", [
    (8, 2, 64),      # even H_k, query group <= 16: two kv heads per unit, 64-key tiles
    (8, 1, 128),     # odd H_k: one kv head per unit
    (64, 2, 128),    # query group of 32: one kv head per unit
])
def test_gen_workspace_size(fm, H, H_k, keys_per_tile):
    # fp32 partial O then (256-byte aligned) LSE, ceil(S_max / keys per tile) + 1
    # slots per (sequence, head)
    B, S_max = 3, 1000
    slots = B * H * ((S_max + keys_per_tile - 1) // keys_per_tile + 1)
    o_bytes = slots * 128 * 4
    assert fm.fmha_gen_workspace_size(B, H, H_k, 128, S_max) == (o_bytes + 255) // 256 * 256 + slots * 4


def call_bwd(fm, **kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, B=2, H=4, Sq=128, Sk=128, D=128, scale=0.1,
             mask=0, ct=0, ws=P, ws_bytes=1 << 30, dt=1, gdt=None)
    a.update(kw)
    gdt = a["dt"] if a["gdt"] is None else a["gdt"]
    t = lambda x: fm.fmha_tensor(a[x], gdt if x in ("dq", "dk", "dv") else a["dt"])
    return fm.lib().fmha_bwd(t("q"), t("k"), t("v"), t("o"), t("do"), a["lse"], t("dq"), t("dk"), t("dv"),
                             a["B"], a["H"], a["Sq"], a["Sk"], a["D"], a["scale"], a["mask"], a["ct"], a["ws"],
                             a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=32), -1), (dict(D=96), -1), (dict(H=0), -1), (dict(B=-1), -1), (dict(Sq=-1), -1),
    (dict(scale=0.0), -1), (dict(scale=float("nan")), -1), (dict(mask=3), -1), (dict(ct=2), -1),
    (dict(q=None), -1), (dict(lse=None), -1), (dict(dk=None), -1), (dict(ws=None), -1), (dict(ws_bytes=16), -1),
    (dict(ws=P + 16), -1), (dict(dt=2), -2), (dict(q=P + 8), -2), (dict(lse=P + 2), -1),
    (dict(dt=2, gdt=0), -2),                          # e4m3 inputs take bf16 gradients
    (dict(dt=2, gdt=1, ws_bytes=2 * 2 * 4 * 128 * 4), -1),   # the 16-bit workspace is too small for e4m3
    (dict(dt=5), -2),
])
def test_bwd_validation_rejects_before_any_launch(fm, kw, code):
    assert call_bwd(fm, **kw) == code


def test_bwd_workspace_size(fm):
    # two fp32 vectors per (b, h), each padded to a multiple of 128 rows
    assert fm.fmha_bwd_workspace_size(2, 4, 100) == 2 * 2 * 4 * 128 * 4
    assert fm.fmha_bwd_workspace_size(1, 3, 300) == 2 * 1 * 3 * 384 * 4
    assert fm.fmha_bwd_workspace_size(0, 4, 100) == 0
    assert call_bwd(fm, B=0) == 0


def test_bwd_workspace_size_ex(fm):
    # 16-bit inputs: as fmha_bwd_workspace_size; e4m3: then 256-byte aligned bf16
    # copies of q, o, dout (B*Sq*H*D each) and k, v (B*Sk*H*D each)
    B, H, Sq, Sk, D = 2, 3, 100, 300, 64
    base = fm.fmha_bwd_workspace_size(B, H, Sq)
    assert fm.fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, 1) == base
    assert fm.fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, 0) == base
    a = lambda x: (x + 255) // 256 * 256
    qb, kb = B * Sq * H * D * 2, B * Sk * H * D * 2
    assert fm.fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, 2) == a(base) + 3 * a(qb) + a(kb) + kb
    assert fm.fmha_bwd_workspace_size_ex(B, H, Sq, Sk, 32, 2) == 0
    assert fm.fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, 7) == 0
