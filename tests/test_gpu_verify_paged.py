"""GPU parity of verify and decode over paged caches (a page pool per key and value, a page
table per sequence): bit-identical to the same sequences over contiguous caches, within
the tolerance of the oracle, and an out-of-pool page entry recorded without a fault."""
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


def _contiguous(seed, lens, rows, cap):
    """Prepared key caches and value caches [n, cap, 2, 256] on the device, fused rows."""
    n = len(lens)
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1)
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1)
    k = torch.stack([synth.normal_bf16(seed, "k", (cap, 2, 256), sub=b) for b in range(n)])
    v = torch.stack([synth.normal_bf16(seed, "v", (cap, 2, 256), sub=b) for b in range(n)])
    qg = torch.stack([synth.normal_bf16(seed, "qg", (rows, 24, 512), sub=b) for b in range(n)])
    c, s = B.ga_rope_table_host(cap)
    c, s = c.cuda(), s.cuda()
    kd = torch.empty_like(k, device="cuda")
    for b in range(n):
        B.ga_k_prologue(k[b].cuda(), w_k.cuda(), c, s, k_prep=kd[b])
    return qg.cuda(), kd, v.cuda(), w_q.cuda(), w_k, (c, s)


def _paginate(kd, vd, lens, rows, page_size, seed, spare=3, max_pages=None):
    """The caches' pages scattered over pools in a random order, with spare pages of other
    finite data; table entries past a sequence's last page are -1 (never read)."""
    n, cap = kd.shape[0], kd.shape[1]
    need = [-(-(L + rows) // page_size) for L in lens]
    total = sum(need) + spare
    rng = np.random.default_rng(seed)
    order = rng.permutation(total)
    kpool = torch.randn(total, page_size, 2, 256, device="cuda").to(torch.bfloat16)
    vpool = torch.randn_like(kpool)
    max_pages = max_pages or max(need)
    table = np.full((n, max_pages), -1, np.int32)
    i = 0
    for b in range(n):
        for p in range(need[b]):
            pg = int(order[i])
            i += 1
            table[b, p] = pg
            lo, hi = p * page_size, min((p + 1) * page_size, cap)
            kpool[pg, :hi - lo] = kd[b, lo:hi]
            vpool[pg, :hi - lo] = vd[b, lo:hi]
    return kpool, vpool, table


@pytest.mark.parametrize("page_size", [128, 256])
@pytest.mark.parametrize("rows", [16, 1])
def test_paged_equals_contiguous_bit_for_bit(page_size, rows):
    """Verify windows (16 rows) and decode (1 row), ragged lengths from 0, windows that end
    inside a page: the paged call gives exactly the contiguous call's bits."""
    lens = [1000, 1537, 0, 383, 128 - rows]
    cap = 1664
    qg, kd, vd, w_q, _, (c, s) = _contiguous(SEED + 40 + rows, lens, rows, cap)
    want = B.ga_attn_verify(qg, kd, vd, lens, w_q, c, s)
    kpool, vpool, table = _paginate(kd, vd, lens, rows, page_size, 41 + page_size)
    pt = torch.from_numpy(table).cuda()
    got = B.ga_attn_verify_paged(qg, kpool, vpool, pt, lens, w_q, c, s)
    torch.cuda.synchronize()
    assert torch.equal(got, want), (got.float() - want.float()).abs().max()


def test_paged_shared_prefix_against_oracle():
    """Two sequences share their first two pages (a common prefix) and then diverge; every
    head against the oracle's gather-then-attend, with the table read through a window of
    more than 32 entries (page size 128, 45 pages for the longer sequence)."""
    rows, page_size = 8, 128
    lens = [5500, 300]
    cap = 5632
    qg, kd, vd, w_q, w_k, (c, s) = _contiguous(SEED + 42, lens, rows, cap)
    kd[1, :256] = kd[0, :256]          # the common prefix: same positions, same keys
    vd[1, :256] = vd[0, :256]
    kpool, vpool, table = _paginate(kd, vd, lens, rows, page_size, 43, max_pages=48)
    table[1, :2] = table[0, :2]        # both sequences read the same two pages
    pt = torch.from_numpy(table).cuda()
    got = B.ga_attn_verify_paged(qg, kpool, vpool, pt, lens, w_q, c, s)
    torch.cuda.synchronize()
    oc, os_ = O.rope_tables(cap)
    kp_np, vp_np = np64(kpool), np64(vpool)
    qg_np, wq_np = np64(qg), np64(w_q)
    heads = [0, 7, 12, 23]
    for b, L in enumerate(lens):
        kc = O.gather_pages(kp_np, table[b], L + rows, page_size)
        vc = O.gather_pages(vp_np, table[b], L + rows, page_size)
        AttnRef(qg_np[b], kc, vc, wq_np, oc, os_, L, L + rows, "causal", heads=heads).check(
            got[b], what=f"paged verify seq {b} L={L}")


def test_paged_out_of_pool_entry_is_recorded_not_a_fault():
    """A page-table entry past the pool (and one negative) is caught by the kernel's own
    bounds check: status 3 in the device status word, zeros read for those tiles, the
    context still usable afterwards."""
    rows, page_size = 4, 128
    lens = [500, 260]
    cap = 640
    qg, kd, vd, w_q, _, (c, s) = _contiguous(SEED + 44, lens, rows, cap)
    kpool, vpool, table = _paginate(kd, vd, lens, rows, page_size, 45)
    n_pages = kpool.shape[0]
    table[0, 1] = n_pages + 5
    table[1, 0] = -7
    pt = torch.from_numpy(table).cuda()
    B.ga_attn_verify_paged(qg, kpool, vpool, pt, lens, w_q, c, s)
    torch.cuda.synchronize()
    assert B.ga_device_status(clear=True) == 3
    assert B.ga_device_status() == 0
    # the same call with a valid table still gives the contiguous bits
    kpool, vpool, table = _paginate(kd, vd, lens, rows, page_size, 45)
    got = B.ga_attn_verify_paged(qg, kpool, vpool, torch.from_numpy(table).cuda(), lens, w_q,
                                 c, s)
    assert torch.equal(got, B.ga_attn_verify(qg, kd, vd, lens, w_q, c, s))
