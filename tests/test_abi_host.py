"""The C ABI without a GPU: the library loads, exports every symbol include/ga_attn.h
declares, validates every argument before any CUDA call, and its host-side RoPE table is
bit-identical to the oracle's.

Refusal tests pass fake pointer values: a refused call never dereferences them (it
returns before any device work), and the library's CUDA-call counter proves it made no
CUDA call at all (system1-omni PR #99: refusals happen before any allocation or CUDA
call; pegainfer PR #1151 review F11: 9 geometry/range refusals, 5 null pointers and 2
zero-length positive controls, device-free).
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def test_exports_every_declared_symbol(L):
    header = open(os.path.join(ROOT, "include", "ga_attn.h")).read()
    names = set(re.findall(r"^\s*(?:int|size_t|const char\*|unsigned long long)\s+(ga_\w+)\s*\(",
                           header, re.M))
    assert names, "no declarations found"
    for n in sorted(names):
        assert hasattr(L, n), n
    assert names == set(B.exported_symbols())


def test_version_geometry_status(L):
    assert B.ga_abi_version() == 1
    assert B.ga_check_geometry() == 0
    assert B.ga_check_geometry(head_dim=128) == -9
    assert B.ga_check_geometry(n_kv_heads=4) == -9
    assert B.ga_check_geometry(rope_base=1e6) == -9
    assert L.ga_check_geometry(None) == -1
    for st in range(-9, 1):
        assert B.ga_status_string(st)
    assert "unknown" in B.ga_status_string(-100)


def test_rope_table_matches_oracle_bit_for_bit(L):
    n = 65552
    c, s = B.ga_rope_table_host(n)
    oc, os_ = O.rope_tables(n)
    assert np.array_equal(c.double().numpy(), oc)
    assert np.array_equal(s.double().numpy(), os_)


# ------------------------------------------------------------------ refusals
A = 0x10000        # a 16-byte-aligned fake device address (never dereferenced)
MIS = 0x10002      # misaligned
S = None           # stream


def _prefill(L, **kw):
    args = dict(qg=A, k=A, v=A, wq=A, cos=A, sin=A, table=8192, rows=128, T=8192, q_base=0,
                causal=1, out=A, stats=None)
    args.update(kw)
    return L.ga_attn_prefill(args["qg"], args["k"], args["v"], args["wq"], args["cos"],
                             args["sin"], args["table"], args["rows"], args["T"],
                             args["q_base"], args["causal"], args["out"], args["stats"], S)


def _masked(L, **kw):
    ws_need = L.ga_masked_workspace_bytes(128, 1024)
    args = dict(qg=A, k=A, v=A, wq=A, cos=A, sin=A, table=1024, rows=128, T=1024, q_base=0,
                mask=A, ld=1024, out=A, w=None, hid=None, ws=0x100000, wsb=ws_need)
    args.update(kw)
    return L.ga_attn_masked(args["qg"], args["k"], args["v"], args["wq"], args["cos"],
                            args["sin"], args["table"], args["rows"], args["T"], args["q_base"],
                            args["mask"], args["ld"], args["out"], args["w"], args["hid"],
                            args["ws"], args["wsb"], S)


def _verify(L, lens=(1000, 2000), **kw):
    n = len(lens)
    arr = (ctypes.c_int * n)(*lens)
    wsb = L.ga_verify_workspace_bytes(n, 16, max(lens))
    args = dict(qg=A, k=A, v=A, cap=4096, arr=arr, n=n, rows=16, wq=A, cos=A, sin=A,
                table=4096, out=A, ws=0x100000, wsb=wsb)
    args.update(kw)
    return L.ga_attn_verify(args["qg"], args["k"], args["v"], args["cap"], args["arr"],
                            args["n"], args["rows"], args["wq"], args["cos"], args["sin"],
                            args["table"], args["out"], args["ws"], args["wsb"], S)


PREFILL_REFUSALS = [
    (dict(qg=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(wq=None), -1),
    (dict(cos=None), -1), (dict(sin=None), -1), (dict(out=None), -1),
    (dict(rows=-1), -2), (dict(T=0), -2), (dict(table=-1), -2),
    (dict(q_base=32, rows=64), -4), (dict(q_base=-64), -4),
    (dict(q_base=8192 - 64, rows=128), -4), (dict(T=(1 << 20) + 1, table=(1 << 20) + 1), -4),
    (dict(causal=0, q_base=64, rows=64), -4), (dict(causal=2), -4),
    (dict(table=127), -5), (dict(q_base=4096, table=4096 + 127), -5),
    (dict(qg=MIS), -3), (dict(k=MIS), -3), (dict(out=MIS), -3), (dict(cos=MIS), -3),
    (dict(stats=MIS + 1), -3),
]


@pytest.mark.parametrize("kw,want", PREFILL_REFUSALS)
def test_prefill_refusals_make_no_cuda_call(L, kw, want):
    before = L.ga_debug_cuda_calls()
    assert _prefill(L, **kw) == want
    assert L.ga_debug_cuda_calls() == before


MASKED_REFUSALS = [
    (dict(mask=None), -1), (dict(T=8193, ld=8208, table=8193), -4), (dict(ld=1000), -4),
    (dict(ld=1036), -3), (dict(mask=MIS), -3), (dict(w=MIS), -3),
    (dict(ws=None), -6), (dict(wsb=100), -6), (dict(ws=0x100010), -6),
    (dict(q_base=64, rows=1024), -4),
]


@pytest.mark.parametrize("kw,want", MASKED_REFUSALS)
def test_masked_refusals_make_no_cuda_call(L, kw, want):
    before = L.ga_debug_cuda_calls()
    assert _masked(L, **kw) == want
    assert L.ga_debug_cuda_calls() == before


def test_verify_refusals_make_no_cuda_call(L):
    cases = [
        (dict(rows=17), -4), (dict(cap=0), -2), (dict(qg=None), -1), (dict(arr=None), -1),
        (dict(table=1000), -5), (dict(ws=None), -6), (dict(wsb=0), -6), (dict(k=MIS), -3),
    ]
    for kw, want in cases:
        before = L.ga_debug_cuda_calls()
        assert _verify(L, **kw) == want, kw
        assert L.ga_debug_cuda_calls() == before
    before = L.ga_debug_cuda_calls()
    assert _verify(L, lens=(1000, 4090)) == -4        # L + rows beyond the cache
    assert _verify(L, lens=(-1, 5)) == -4
    assert L.ga_debug_cuda_calls() == before


def _verify_paged(L, lens=(1000, 2000), **kw):
    n = len(lens)
    arr = (ctypes.c_int * n)(*lens)
    wsb = L.ga_verify_workspace_bytes(n, 16, max(lens, default=0))
    args = dict(qg=A, k=A, v=A, n_pages=40, page_size=256, pt=A, max_pages=16, arr=arr, n=n,
                rows=16, wq=A, cos=A, sin=A, table=4096, out=A, ws=0x100000, wsb=wsb)
    args.update(kw)
    return L.ga_attn_verify_paged(args["qg"], args["k"], args["v"], args["n_pages"],
                                  args["page_size"], args["pt"], args["max_pages"], args["arr"],
                                  args["n"], args["rows"], args["wq"], args["cos"], args["sin"],
                                  args["table"], args["out"], args["ws"], args["wsb"], S)


def test_verify_paged_refusals_make_no_cuda_call(L):
    cases = [
        (dict(pt=None), -1), (dict(k=None), -1), (dict(arr=None), -1),
        (dict(n_pages=0), -2), (dict(page_size=0), -2), (dict(max_pages=0), -2),
        (dict(rows=17), -4), (dict(page_size=200), -4), (dict(page_size=(1 << 20) + 128), -4),
        (dict(max_pages=7), -4),                     # 2000 + 16 positions need 8 pages of 256
        (dict(lens=(5, -1)), -4), (dict(table=1000), -5), (dict(pt=A + 2), -3),
        (dict(v=MIS), -3), (dict(ws=None), -6), (dict(wsb=0), -6),
    ]
    for kw, want in cases:
        before = L.ga_debug_cuda_calls()
        assert _verify_paged(L, **kw) == want, kw
        assert L.ga_debug_cuda_calls() == before
    before = L.ga_debug_cuda_calls()
    assert _verify_paged(L, rows=0, wsb=256) == 0        # an empty call is a no-op
    assert _verify_paged(L, lens=()) == 0
    assert L.ga_debug_cuda_calls() == before


def _batch(L, starts=(0, 300, 300, 1000), bases=(0, 64, 1024), **kw):
    n = len(bases)
    st = (ctypes.c_int * len(starts))(*starts)
    qb = (ctypes.c_int * max(n, 1))(*bases)
    args = dict(qg=A, st=st, qb=qb, n=n, k=A, v=A, n_pages=64, page_size=128, pt=A,
                max_pages=16, wq=A, cos=A, sin=A, table=4096, out=A)
    args.update(kw)
    return L.ga_attn_prefill_batch(args["qg"], args["st"], args["qb"], args["n"], args["k"],
                                   args["v"], args["n_pages"], args["page_size"], args["pt"],
                                   args["max_pages"], args["wq"], args["cos"], args["sin"],
                                   args["table"], args["out"], S)


def test_prefill_batch_refusals_make_no_cuda_call(L):
    cases = [
        (dict(qg=None), -1), (dict(st=None), -1), (dict(pt=None), -1), (dict(out=None), -1),
        (dict(n=-1), -2), (dict(n_pages=0), -2), (dict(max_pages=0), -2),
        (dict(starts=(0, 300, 200, 1000)), -2),          # a sequence with -100 rows
        (dict(starts=(-5, 300, 300, 1000)), -2),
        (dict(bases=(0, 65, 1024)), -4), (dict(bases=(0, -64, 1024)), -4),
        (dict(page_size=192), -4),
        (dict(max_pages=13), -4),                         # 1024 + 700 keys need 14 pages
        (dict(table=1700), -5),                           # the longest window ends at 1724
        (dict(pt=A + 1), -3), (dict(k=MIS), -3), (dict(out=MIS), -3),
    ]
    for kw, want in cases:
        before = L.ga_debug_cuda_calls()
        assert _batch(L, **kw) == want, kw
        assert L.ga_debug_cuda_calls() == before
    before = L.ga_debug_cuda_calls()
    assert _batch(L, starts=(0, 0, 0, 0)) == 0            # no rows: a no-op
    assert _batch(L, starts=(7,), bases=()) == 0           # no sequences
    assert L.ga_debug_cuda_calls() == before


def test_quantize_refusals_make_no_cuda_call(L):
    before = L.ga_debug_cuda_calls()
    assert L.ga_kv_quantize_e4m3(None, 10, A, A, S) == -1
    assert L.ga_kv_quantize_e4m3(A, 10, None, A, S) == -1
    assert L.ga_kv_quantize_e4m3(A, 10, A, None, S) == -1
    assert L.ga_kv_quantize_e4m3(A, -1, A, A, S) == -2
    assert L.ga_kv_quantize_e4m3(A, (1 << 26) + 1, A, A, S) == -4
    assert L.ga_kv_quantize_e4m3(A + 4, 10, A, A, S) == -3
    assert L.ga_kv_quantize_e4m3(A, 10, A + 2, A, S) == -3
    assert L.ga_kv_quantize_e4m3(A, 0, A, A, S) == 0          # no rows: a no-op
    assert L.ga_debug_cuda_calls() == before


def test_select_mask_refusals_make_no_cuda_call(L):
    before = L.ga_debug_cuda_calls()
    f = L.ga_select_mask
    assert f(None, 2048, 10, 8192, 0, 512, A, 8192, S) == -1
    assert f(A, 2048, 10, 8192, 0, 512, None, 8192, S) == -1
    assert f(A, 2048, -1, 8192, 0, 512, A, 8192, S) == -2
    assert f(A, 2048, 10, 0, 0, 512, A, 8192, S) == -2
    assert f(A, 2048, 10, 8192, -1, 512, A, 8192, S) == -2
    assert f(A, 2048, 10, 8192, 0, 0, A, 8192, S) == -2
    assert f(A, 2049, 10, 8196, 0, 512, A, 8208, S) == -4       # T over the masked cap
    assert f(A, 2048, 10, 8192, 8183, 512, A, 8192, S) == -4    # q_base + rows > T
    assert f(A, 2047, 10, 8192, 0, 512, A, 8192, S) == -4       # ld_scores < ceil(T / 4)
    assert f(A, 26, 10, 101, 0, 4, A, 96, S) == -4              # ld_mask < T
    assert f(A, 1 << 32, 10, 8192, 0, 4, A, 8192, S) == -4
    assert f(A, 2048, 10, 8192, 0, 512, A, 8200, S) == -3       # ld_mask % 16
    assert f(A, 2048, 10, 8192, 0, 512, A + 8, 8192, S) == -3
    assert f(A + 2, 2048, 10, 8192, 0, 512, A, 8192, S) == -3
    assert f(A, 2048, 0, 8192, 0, 512, A, 8192, S) == 0         # no rows: a no-op
    assert f(A, 26, 10, 101, 91, 4, A + 4, 112, S) == -3
    assert L.ga_debug_cuda_calls() == before


def test_dequantize_and_prefill_e4m3_refusals_make_no_cuda_call(L):
    before = L.ga_debug_cuda_calls()
    f = L.ga_kv_dequantize_e4m3
    assert f(None, A, 10, A, S) == -1
    assert f(A, None, 10, A, S) == -1
    assert f(A, A, 10, None, S) == -1
    assert f(A, A, -1, A, S) == -2
    assert f(A, A, (1 << 26) + 1, A, S) == -4
    assert f(A + 4, A, 10, A, S) == -3
    assert f(A, A + 2, 10, A, S) == -3
    assert f(A, A, 10, A + 8, S) == -3
    assert f(A, A, 0, A, S) == 0                       # no rows: a no-op
    assert L.ga_prefill_e4m3_workspace_bytes(0) == 0
    assert L.ga_prefill_e4m3_workspace_bytes(1000) == 2 * 1000 * 2 * 256 * 2
    ws = L.ga_prefill_e4m3_workspace_bytes(512)
    g = L.ga_attn_prefill_e4m3
    ok = (A, A, A, A, A, A, A, A, 512, 128, 512, 0, 1, A, None, A, ws, S)
    def call(**kw):
        names = ["qg", "kc", "ks", "vc", "vs", "wq", "cos", "sin", "tr", "rows", "T", "qb",
                 "causal", "out", "rs", "ws", "wsb", "s"]
        args = dict(zip(names, ok))
        args.update(kw)
        return g(*[args[n] for n in names])
    assert call(kc=None) == -1
    assert call(vs=None) == -1
    assert call(rows=-1) == -2
    assert call(qb=32) == -4                           # q_base not a multiple of 64
    assert call(causal=2) == -4
    assert call(qb=64, rows=64, causal=0) == -4        # bidirectional starts at 0
    assert call(tr=100) == -5
    assert call(kc=A + 8) == -3                        # codes 16-byte aligned
    assert call(ks=A + 2) == -3
    assert call(ws=None) == -6
    assert call(ws=A + 16) == -6
    assert call(wsb=ws - 1) == -6
    assert call(rows=0) == 0                           # no rows: a no-op
    assert L.ga_debug_cuda_calls() == before


def test_k_prologue_refusals(L):
    before = L.ga_debug_cuda_calls()
    assert L.ga_k_prologue(None, A, A, A, 100, 10, 0, A, S) == -1
    assert L.ga_k_prologue(A, A, A, A, 100, -1, 0, A, S) == -2
    assert L.ga_k_prologue(A, A, A, A, 100, 10, -1, A, S) == -4
    assert L.ga_k_prologue(A, A, A, A, 100, 10, 95, A, S) == -5
    assert L.ga_k_prologue(A, A, A, A, 100, 10, 0, MIS, S) == -3
    assert L.ga_debug_cuda_calls() == before


def test_qk_prologue_refusals(L):
    """Both prologues in one launch: every argument check of the two single calls, before any
    CUDA call. Arguments: k_raw, w_k, n_tok, k_pos_base, k_prep, qg, w_q, rows, q_base,
    q_prep, cos, sin, table_rows, stream."""
    before = L.ga_debug_cuda_calls()
    Q = L.ga_qk_prologue
    assert Q(None, A, 10, 0, A, A, A, 10, 0, A, A, A, 100, S) == -1
    assert Q(A, A, 10, 0, A, A, A, 10, 0, None, A, A, 100, S) == -1
    assert Q(A, A, -1, 0, A, A, A, 10, 0, A, A, A, 100, S) == -2
    assert Q(A, A, 10, 0, A, A, A, -1, 0, A, A, A, 100, S) == -2
    assert Q(A, A, 10, -1, A, A, A, 10, 0, A, A, A, 100, S) == -4
    assert Q(A, A, 10, 0, A, A, A, 10, -1, A, A, A, 100, S) == -4
    assert Q(A, A, 10, 95, A, A, A, 10, 0, A, A, A, 100, S) == -5   # key positions past the table
    assert Q(A, A, 10, 0, A, A, A, 10, 95, A, A, A, 100, S) == -5   # query positions past it
    assert Q(MIS, A, 10, 0, A, A, A, 10, 0, A, A, A, 100, S) == -3
    assert Q(A, A, 10, 0, A, A, A, 10, 0, MIS, A, A, 100, S) == -3
    assert Q(A, A, 10, 0, A, A, MIS, 10, 0, A, A, A, 100, S) == -3
    assert Q(A, A, 0, 0, A, A, A, 0, 0, A, A, A, 100, S) == 0      # nothing to do
    assert L.ga_debug_cuda_calls() == before


def test_q_prologue_and_prepared_refusals(L):
    before = L.ga_debug_cuda_calls()
    assert L.ga_q_prologue(None, A, A, A, 100, 10, 0, A, S) == -1
    assert L.ga_q_prologue(A, A, A, A, 100, -1, 0, A, S) == -2
    assert L.ga_q_prologue(A, A, A, A, 100, 10, -1, A, S) == -4
    assert L.ga_q_prologue(A, A, A, A, 100, 10, 95, A, S) == -5
    assert L.ga_q_prologue(A, A, A, A, 100, 10, 0, MIS, S) == -3
    P = L.ga_attn_prefill_prepared
    assert P(None, A, A, A, 10, 100, 0, 1, A, None, S) == -1
    assert P(A, A, A, A, -1, 100, 0, 1, A, None, S) == -2
    assert P(A, A, A, A, 10, 100, 32, 1, A, None, S) == -4      # q_base not a multiple of 64
    assert P(A, A, A, A, 10, 100, 64, 0, A, None, S) == -4      # bidirectional window
    assert P(A, A, A, A, 200, 100, 0, 1, A, None, S) == -4      # rows beyond T
    assert P(A, A, A, A, 10, 100, 0, 2, A, None, S) == -4
    assert P(MIS, A, A, A, 10, 100, 0, 1, A, None, S) == -3
    assert P(A, A, A, A, 10, 100, 0, 1, A, MIS + 1, S) == -3
    assert L.ga_debug_cuda_calls() == before


def test_masked_prepared_refusals(L):
    before = L.ga_debug_cuda_calls()
    P = L.ga_attn_masked_prepared
    wsb = L.ga_masked_workspace_bytes(10, 100)
    W = 0x20000                                             # 256-byte aligned fake workspace
    assert P(None, A, A, A, 10, 100, 0, A, 112, A, None, None, W, wsb, S) == -1
    assert P(A, A, A, A, 10, 100, 0, None, 112, A, None, None, W, wsb, S) == -1
    assert P(A, A, A, A, -1, 100, 0, A, 112, A, None, None, W, wsb, S) == -2
    assert P(A, A, A, A, 10, 100, 32, A, 112, A, None, None, W, wsb, S) == -4
    assert P(A, A, A, A, 10, 9000, 0, A, 9008, A, None, None, W, wsb, S) == -4   # masked cap
    assert P(A, A, A, A, 10, 100, 0, A, 96, A, None, None, W, wsb, S) == -4      # ld < T
    assert P(MIS, A, A, A, 10, 100, 0, A, 112, A, None, None, W, wsb, S) == -3
    assert P(A, A, A, A, 10, 100, 0, A, 104, A, None, None, W, wsb, S) == -3     # ld % 16
    assert P(A, A, A, A, 10, 100, 0, A, 112, A, None, None, W, wsb - 1, S) == -6
    assert P(A, A, A, A, 10, 100, 0, A, 112, A, None, None, W + 16, wsb, S) == -6
    assert P(A, A, A, A, 0, 100, 0, A, 112, A, None, None, W, wsb, S) == 0        # no-op
    assert L.ga_debug_cuda_calls() == before


def test_kv_group_refusals(L):
    before = L.ga_debug_cuda_calls()
    P = L.ga_attn_prefill_kv
    for first, count in [(-1, 1), (0, 0), (1, 2), (2, 1), (0, 3)]:
        assert P(A, A, A, A, A, A, 100, 10, 100, 0, 1, first, count, A, None, S) == -4
    assert P(None, A, A, A, A, A, 100, 10, 100, 0, 1, 0, 1, A, None, S) == -1
    assert P(A, A, A, A, A, A, 100, 0, 100, 0, 1, 1, 1, A, None, S) == 0          # no-op
    M = L.ga_attn_masked_kv
    wsb = L.ga_masked_workspace_bytes(10, 100)
    W = 0x20000
    for first, count in [(-1, 1), (0, 0), (1, 2)]:
        assert M(A, A, A, A, A, A, 100, 10, 100, 0, A, 112, first, count, A, None, None, W, wsb,
                 S) == -4
    assert M(A, A, A, A, A, A, 100, 10, 100, 0, A, 112, 1, 1, A, None, None, W, wsb - 1, S) == -6
    assert M(A, A, A, A, A, A, 100, 0, 100, 0, A, 112, 1, 1, A, None, None, W, wsb, S) == 0
    assert L.ga_debug_cuda_calls() == before


def test_qk_probe_refusals(L):
    before = L.ga_debug_cuda_calls()
    assert L.ga_debug_qk_fp32(None, A, 1, A, S) == -1
    assert L.ga_debug_qk_fp32(A, A, -1, A, S) == -2
    assert L.ga_debug_qk_fp32(A, A, 70000, A, S) == -4
    assert L.ga_debug_qk_fp32(A, MIS, 1, A, S) == -3
    assert L.ga_debug_qk_fp32(A, A, 0, A, S) == 0
    assert L.ga_debug_cuda_calls() == before


def test_pair_switch(L):
    """The form switch makes no CUDA call: modes 0, 1 and 2 round-trip, the rest are
    refused with RANGE and leave the mode as it was."""
    before = L.ga_debug_cuda_calls()
    mode = L.ga_debug_set_cta_pairs(0)
    assert mode in (0, 1, 2)
    assert L.ga_debug_set_cta_pairs(3) == -4 and L.ga_debug_set_cta_pairs(-1) == -4
    assert L.ga_debug_set_cta_pairs(2) == 0
    assert L.ga_debug_set_cta_pairs(mode) == 2
    assert L.ga_debug_cuda_calls() == before


def test_wait_timeout_hook_refuses_bad_limits(L):
    before = L.ga_debug_cuda_calls()
    assert L.ga_debug_wait_timeout(0, S) == -4
    assert L.ga_debug_wait_timeout(3_000_000_000, S) == -4
    assert L.ga_debug_cuda_calls() == before


def test_empty_calls_are_noops_without_cuda(L):
    before = L.ga_debug_cuda_calls()
    assert _prefill(L, rows=0) == 0
    assert _masked(L, rows=0, wsb=L.ga_masked_workspace_bytes(0, 1024)) == 0
    assert _verify(L, rows=0, wsb=256) == 0
    assert L.ga_k_prologue(A, A, A, A, 100, 0, 0, A, S) == 0
    assert L.ga_q_prologue(A, A, A, A, 100, 0, 0, A, S) == 0
    assert L.ga_attn_prefill_prepared(A, A, A, A, 0, 100, 0, 1, A, None, S) == 0
    assert L.ga_debug_cuda_calls() == before


def test_workspace_sizes(L):
    # bit mask, tile flags, row statistics and the prepared queries
    assert L.ga_masked_workspace_bytes(8192, 8192) >= (8192 * 256 * 4 + 64 * 64 + 24 * 8192 * 8
                                                       + 8192 * 6144 * 2)
    assert L.ga_masked_workspace_bytes(1, 8193) == 0
    assert L.ga_masked_workspace_bytes(-1, 10) == 0
    assert L.ga_verify_workspace_bytes(0, 16, 10) == 0
