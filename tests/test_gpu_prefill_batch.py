"""GPU parity of the batched causal prefill over paged caches: every sequence of a batch
gives the one-sequence entry point's bits, branches that share a prefix's pages give the
full pass's rows, a sequence longer than one launch's tables is cut into windows without a
trace in the results, and sampled heads meet the oracle."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, AttnRef, np64
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod
from verify_gated_gqa_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.lib()
    yield
    assert B.ga_device_status() == 0


def _sequence(seed, sub, T, w_k, c, s):
    """Prepared keys and values of positions 0 .. T-1 of one sequence, on the device."""
    k = synth.normal_bf16(seed, "k", (T, 2, 256), sub=sub, device="cuda")
    v = synth.normal_bf16(seed, "v", (T, 2, 256), sub=sub, device="cuda")
    kd = torch.empty_like(k)
    if T:
        B.ga_k_prologue(k, w_k, c, s, k_prep=kd)
    return kd, v


def _pages(caches, page_size, seed, spare=2):
    """Scatter each cache (a list of [T_b, 2, 256] key/value pairs) over two pools in a
    random page order; spare pages hold other finite data; unused table entries are -1."""
    need = [-(-kd.shape[0] // page_size) for kd, _ in caches]
    total = sum(need) + spare
    order = np.random.default_rng(seed).permutation(total)
    kpool = torch.randn(total, page_size, 2, 256, device="cuda").to(torch.bfloat16)
    vpool = torch.randn_like(kpool)
    table = np.full((len(caches), max(max(need), 1)), -1, np.int32)
    i = 0
    for b, (kd, vd) in enumerate(caches):
        for p in range(need[b]):
            pg = int(order[i])
            i += 1
            table[b, p] = pg
            lo, hi = p * page_size, min((p + 1) * page_size, kd.shape[0])
            kpool[pg, :hi - lo] = kd[lo:hi]
            vpool[pg, :hi - lo] = vd[lo:hi]
    return kpool, vpool, table


def _setup(seed, spec, table_rows):
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1, device="cuda")
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1, device="cuda")
    c, s = B.ga_rope_table_host(table_rows)
    c, s = c.cuda(), s.cuda()
    caches = [_sequence(seed, b, qb + rows, w_k, c, s) for b, (qb, rows) in enumerate(spec)]
    qgs = [synth.normal_bf16(seed, "qg", (rows, 24, 512), sub=b, device="cuda")
           for b, (qb, rows) in enumerate(spec)]
    starts = np.concatenate([[0], np.cumsum([rows for _, rows in spec])]).astype(int)
    return w_q, (c, s), caches, qgs, starts


@pytest.mark.parametrize("page_size", [128, 256])
def test_batch_equals_one_sequence_calls(page_size):
    """Windows at q_base 0, 64, 1024, 128 and 256, an empty sequence and a one-row one: each
    sequence's rows equal ga_attn_prefill's over the same keys, bit for bit."""
    spec = [(0, 300), (64, 129), (1024, 700), (0, 1), (128, 0), (256, 128)]
    w_q, (c, s), caches, qgs, starts = _setup(SEED + 50, spec, 2048)
    kpool, vpool, table = _pages(caches, page_size, 51 + page_size)
    qg = torch.cat(qgs)
    got = B.ga_attn_prefill_batch(qg, starts, [qb for qb, _ in spec], kpool, vpool,
                                  torch.from_numpy(table).cuda(), w_q, c, s)
    for b, (qb, rows) in enumerate(spec):
        if rows == 0:
            continue
        kd, vd = caches[b]
        want = B.ga_attn_prefill(qgs[b], kd, vd, w_q, c, s, qb, qb + rows)
        assert torch.equal(got[starts[b]:starts[b + 1]], want), f"sequence {b} {spec[b]}"


def test_batch_branches_share_a_prefix():
    """A 256-token prefix (two pages of 128) and three branches of 1, 70 and 200 tokens
    whose page-table rows list the prefix's pages and then their own: each branch's rows
    equal rows 256.. of a full causal pass over prefix + branch; the prefix runs in the same
    batch."""
    P, page = 256, 128
    branches = [1, 70, 200]
    seed = SEED + 52
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1, device="cuda")
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1, device="cuda")
    c, s = B.ga_rope_table_host(P + max(branches))
    c, s = c.cuda(), s.cuda()
    k_pre = synth.normal_bf16(seed, "k", (P, 2, 256), device="cuda")
    v_pre = synth.normal_bf16(seed, "v", (P, 2, 256), device="cuda")
    kd_pre = torch.empty_like(k_pre)
    B.ga_k_prologue(k_pre, w_k, c, s, k_prep=kd_pre)
    qg_pre = synth.normal_bf16(seed, "qg", (P, 24, 512), device="cuda")
    n_br = len(branches)
    n_pages = 2 + sum(-(-n // page) for n in branches)
    kpool = torch.zeros(n_pages, page, 2, 256, dtype=torch.bfloat16, device="cuda")
    vpool = torch.zeros_like(kpool)
    kpool[0], kpool[1] = kd_pre[:128], kd_pre[128:]
    vpool[0], vpool[1] = v_pre[:128], v_pre[128:]
    table = np.full((1 + n_br, 4), -1, np.int32)
    table[:, :2] = [0, 1]
    nxt = 2
    full_k, full_v, qgs = [], [], [qg_pre]
    for i, n in enumerate(branches):
        k_br = synth.normal_bf16(seed, "k", (n, 2, 256), sub=i + 1, device="cuda")
        v_br = synth.normal_bf16(seed, "v", (n, 2, 256), sub=i + 1, device="cuda")
        kd_br = torch.empty_like(k_br)
        B.ga_k_prologue(k_br, w_k, c, s, pos_base=P, k_prep=kd_br)
        for p in range(-(-n // page)):
            lo, hi = p * page, min((p + 1) * page, n)
            kpool[nxt, :hi - lo] = kd_br[lo:hi]
            vpool[nxt, :hi - lo] = v_br[lo:hi]
            table[1 + i, 2 + p] = nxt
            nxt += 1
        full_k.append(torch.cat([kd_pre, kd_br]))
        full_v.append(torch.cat([v_pre, v_br]))
        qgs.append(synth.normal_bf16(seed, "qg", (n, 24, 512), sub=i + 1, device="cuda"))
    starts = np.concatenate([[0], np.cumsum([P] + branches)]).astype(int)
    got = B.ga_attn_prefill_batch(torch.cat(qgs), starts, [0] + [P] * n_br, kpool, vpool,
                                  torch.from_numpy(table).cuda(), w_q, c, s)
    want_pre = B.ga_attn_prefill(qg_pre, kd_pre, v_pre, w_q, c, s, 0, P)
    assert torch.equal(got[:P], want_pre)
    for i, n in enumerate(branches):
        full = B.ga_attn_prefill(torch.cat([qg_pre, qgs[1 + i]]), full_k[i], full_v[i], w_q,
                                 c, s, 0, P + n)
        assert torch.equal(got[starts[1 + i]:starts[2 + i]], full[P:]), f"branch {i}"


def test_batch_sequence_longer_than_one_launch():
    """32,968 rows (more than 256 row tiles) in one sequence: the call cuts it into a
    32,768-row window and a 200-row window at q_base 32,768; the result equals the
    one-sequence pass bit for bit."""
    rows, page = 32768 + 200, 256
    spec = [(0, rows)]
    w_q, (c, s), caches, qgs, starts = _setup(SEED + 53, spec, rows)
    kpool, vpool, table = _pages(caches, page, 54, spare=0)
    got = B.ga_attn_prefill_batch(qgs[0], starts, [0], kpool, vpool,
                                  torch.from_numpy(table).cuda(), w_q, c, s)
    kd, vd = caches[0]
    want = B.ga_attn_prefill(qgs[0], kd, vd, w_q, c, s, 0, rows)
    assert torch.equal(got, want)


def test_batch_against_oracle():
    """Sampled heads of three sequences against the oracle over the gathered pages."""
    spec = [(0, 200), (192, 64), (640, 130)]
    w_q, (c, s), caches, qgs, starts = _setup(SEED + 55, spec, 1024)
    page = 128
    kpool, vpool, table = _pages(caches, page, 56)
    got = B.ga_attn_prefill_batch(torch.cat(qgs), starts, [qb for qb, _ in spec], kpool, vpool,
                                  torch.from_numpy(table).cuda(), w_q, c, s)
    torch.cuda.synchronize()
    oc, os_ = O.rope_tables(1024)
    kp_np, vp_np, wq_np = np64(kpool), np64(vpool), np64(w_q)
    heads = [0, 5, 12, 23]
    for b, (qb, rows) in enumerate(spec):
        T = qb + rows
        kc = O.gather_pages(kp_np, table[b], T, page)
        vc = O.gather_pages(vp_np, table[b], T, page)
        AttnRef(np64(qgs[b]), kc, vc, wq_np, oc, os_, qb, T, "causal", heads=heads).check(
            got[starts[b]:starts[b + 1]], what=f"batch seq {b} (q_base {qb}, {rows} rows)")


@pytest.mark.parametrize("page_size", [128, 256])
def test_batch_pairs_equal_single(page_size):
    """The batched pass as CTA pairs (half K/V tiles per CTA from the paged pools, output tiles
    by TMA stores where a sequence fills them, the rows' own stores where it ends inside one)
    against single CTAs: the same bits, on windows at several positions, an empty sequence,
    one row and tiles that end mid-sequence."""
    spec = [(0, 300), (64, 129), (1024, 700), (0, 1), (128, 0), (256, 128), (0, 256)]
    w_q, (c, s), caches, qgs, starts = _setup(SEED + 52, spec, 2048)
    kpool, vpool, table = _pages(caches, page_size, 53 + page_size)
    qg = torch.cat(qgs)
    tab = torch.from_numpy(table).cuda()
    outs = []
    for pairs in (False, True):
        prev = B.ga_debug_set_cta_pairs(2 if pairs else 0)
        try:
            outs.append(B.ga_attn_prefill_batch(qg, starts, [qb for qb, _ in spec], kpool, vpool,
                                                tab, w_q, c, s))
            torch.cuda.synchronize()
        finally:
            B.ga_debug_set_cta_pairs(prev)
    assert B.ga_device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
