"""GPU parity of the few-row verify windows against the oracle and against the prefill
entry point (the same rows over the same keys)."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import compare, SEED, AttnRef, np64
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


def _verify_case(seed, lens, rows, cap):
    """Per sequence: raw keys/values of positions 0..cap-1, qg rows at positions L..L+rows-1."""
    n = len(lens)
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1)
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1)
    k = torch.stack([synth.normal_bf16(seed, "k", (cap, 2, 256), sub=b) for b in range(n)])
    v = torch.stack([synth.normal_bf16(seed, "v", (cap, 2, 256), sub=b) for b in range(n)])
    qg = torch.stack([synth.normal_bf16(seed, "qg", (rows, 24, 512), sub=b) for b in range(n)])
    return qg, k, v, w_q, w_k


def _run(seed, lens, rows, cap):
    qg, k, v, w_q, w_k = _verify_case(seed, lens, rows, cap)
    c, s = B.ga_rope_table_host(cap)
    c, s = c.cuda(), s.cuda()
    kd = torch.empty_like(k, device="cuda")
    for b in range(len(lens)):
        B.ga_k_prologue(k[b].cuda(), w_k.cuda(), c, s, k_prep=kd[b])
    out = B.ga_attn_verify(qg.cuda(), kd, v.cuda(), lens, w_q.cuda(), c, s)
    return out, (qg, k, v, w_q, w_k), kd, (c, s)


def _refs(data, lens, cap, heads=None):
    """Oracle per sequence: row r at position L_b + r over prepared keys 0 .. L_b + r."""
    qg, k, v, w_q, w_k = [np64(x) for x in data]
    oc, os_ = O.rope_tables(cap)
    res = {}
    for b in range(len(lens)):
        kp = O.prep_keys(k[b], w_k, oc, os_)
        L = lens[b]
        res[b] = AttnRef(qg[b], kp, v[b], w_q, oc, os_, L, L + qg.shape[1], "causal",
                         heads=heads)
    return res


def test_verify_small_all_heads():
    lens, rows, cap = [1000, 1537, 0], 16, 1600
    out, data, kd, (c, s) = _run(SEED + 30, lens, rows, cap)
    refs = _refs(data, lens, cap)
    for b in range(len(lens)):
        refs[b].check(out[b], what=f"verify seq {b} L={lens[b]}")


def test_verify_equals_prefill_rows():
    lens, rows, cap = [700, 1283], 16, 1300
    out, data, kd, (c, s) = _run(SEED + 31, lens, rows, cap)
    qg, k, v, w_q, w_k = data
    for b, L in enumerate(lens):
        # prefill over the same keys: the window's rows at q_base = L need L % 64 == 0 for
        # the prefill entry point, so compare through a 64-aligned window that ends at L+rows
        qb = (L // 64) * 64
        T = L + rows
        qg_full = torch.cat([synth.normal_bf16(0, "qg", (L - qb, 24, 512)), qg[b]]).cuda()
        ref = B.ga_attn_prefill(qg_full, kd[b], v[b].cuda(), w_q.cuda(), c, s, qb, T)
        # the split-key partials are summed in another fp32 order than the single pass, so
        # the two agree within the stated tolerance rather than bit for bit
        st = compare(out[b], np64(ref[L - qb:]))
        print(f"[info] verify vs prefill rows, seq {b}: {st}")
        assert st["bad"] == 0 and st["nan"] == 0, st


def test_verify_long_cache_sampled():
    """The long-cache verify shape on two sequences: 16 rows at positions 65,536..65,551 over 65,536
    cached keys (cap 65,552); sampled heads against the oracle."""
    lens, rows, cap = [65536, 65536], 16, 65552
    out, data, kd, _ = _run(SEED + 32, lens, rows, cap)
    heads = [0, 11, 12, 23]
    refs = _refs(data, lens, cap, heads=heads)
    for b in range(2):
        refs[b].check(out[b], what=f"verify L=65536 seq {b} heads {heads}")


def test_verify_one_sequence_l65536_many_chunks():
    """One sequence of 16 rows over 65,536 cached keys: the launch splits its keys into 37
    chunks (more than one warp's lanes), so the combine reads its (M, l) pairs from two lanes
    per row and sums the partial rows four chunks at a time; sampled heads against the
    oracle."""
    lens, rows, cap = [65536], 16, 65552
    out, data, kd, _ = _run(SEED + 35, lens, rows, cap)
    heads = [0, 13, 23]
    _refs(data, lens, cap, heads=heads)[0].check(out[0], what=f"verify L=65536, one sequence, "
                                                             f"heads {heads}")


def test_verify_8x16_l65536_launch_sampled():
    """The benchmark's launch: 8 sequences x 16 rows at positions 65,536..65,551 over caches
    of 65,552 positions (the chunking the bench times); two sequences' sampled heads
    against the oracle, which prepares its own keys from the raw ones."""
    lens, rows, cap, n = [65536] * 8, 16, 65552, 8
    seed = SEED + 35
    dev = "cuda"
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1)
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1)
    c, s = B.ga_rope_table_host(cap)
    c, s = c.cuda(), s.cuda()
    kd = torch.empty(n, cap, 2, 256, dtype=torch.bfloat16, device=dev)
    vd = torch.empty_like(kd)
    sampled = (0, 7)
    raw = {}
    for b in range(n):
        if b in sampled:
            k_raw = synth.normal_bf16(seed, "k", (cap, 2, 256), sub=b)
            v_raw = synth.normal_bf16(seed, "v", (cap, 2, 256), sub=b)
            raw[b] = (k_raw, v_raw)
            k_dev, vd[b] = k_raw.to(dev), v_raw.to(dev)
        else:
            k_dev = synth.normal_bf16(seed, "k", (cap, 2, 256), sub=b, device=dev)
            vd[b] = synth.normal_bf16(seed, "v", (cap, 2, 256), sub=b, device=dev)
        B.ga_k_prologue(k_dev, w_k.to(dev), c, s, k_prep=kd[b])
    qg = torch.stack([synth.normal_bf16(seed, "qg", (rows, 24, 512), sub=b) for b in range(n)])
    out = B.ga_attn_verify(qg.to(dev), kd, vd, lens, w_q.to(dev), c, s)
    torch.cuda.synchronize()
    oc, os_ = O.rope_tables(cap)
    heads = [3, 12, 22]
    for b in sampled:
        k_hat = O.prep_keys(np64(raw[b][0]), np64(w_k), oc, os_)
        AttnRef(np64(qg[b]), k_hat, np64(raw[b][1]), np64(w_q), oc, os_, lens[b],
                lens[b] + rows, "causal", heads=heads).check(
            out[b], what=f"verify 8 x 16 rows at L=65536, seq {b}, heads {heads}")


def test_verify_single_sequence():
    """One sequence per call, 7 rows (the key/value map keeps its sequence dimension)."""
    lens, rows, cap = [900], 7, 912
    out, data, kd, _ = _run(SEED + 33, lens, rows, cap)
    _refs(data, lens, cap)[0].check(out[0], what="verify, one sequence of 7 rows")


def test_verify_65_sequences_two_groups():
    """65 sequences of 4 rows: one launch for the first 64 sequences and one for the last
    alone; ragged lengths from 0 to 299 (including L = 0)."""
    n = 65
    rng = np.random.default_rng(34)
    lens = [int(x) for x in rng.integers(0, 300, n)]
    lens[5] = 0
    rows, cap = 4, 320
    out, data, kd, _ = _run(SEED + 34, lens, rows, cap)
    for b in (0, 5, 31, 63, 64):
        sub = tuple(x[b:b + 1] for x in data[:3]) + tuple(data[3:])
        _refs(sub, [lens[b]], cap)[0].check(out[b], what=f"verify, 65 sequences, seq {b}")
