"""GPU parity of the K prologue and the causal / window / bidirectional attention against
the CPU oracle, through the C ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, Inputs, compare, np64
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod
from verify_gated_gqa_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.lib()
    assert torch.cuda.is_available()
    yield
    assert B.ga_device_status() == 0


def _oracle_prefill(inp, q_base, T, causal, rows=None, heads=None, mode="R1", qg=None):
    c, s = inp.oracle_tables(mode)
    kp = O.prep_keys(inp.np["k"], inp.np["w_k"], c, s, mode=mode)
    qg = inp.np["qg"] if qg is None else qg
    return O.prefill(qg, kp, inp.np["v"], inp.np["w_q"], c, s, q_base, T, causal, mode,
                     rows=rows, heads=heads)


# ------------------------------------------------------------------ K prologue
@pytest.mark.parametrize("T,pos_base", [(2048, 0), (333, 777)])
def test_k_prologue_bit_exact(T, pos_base):
    inp = Inputs(SEED + 7, 1, T)
    c, s = B.ga_rope_table_host(pos_base + T)
    d = inp.dev()
    got = B.ga_k_prologue(d["k"], d["w_k"], c.cuda(), s.cuda(), pos_base=pos_base)
    oc, os_ = O.rope_tables(pos_base + T)
    want = O.prep_keys(inp.np["k"], inp.np["w_k"], oc, os_, pos0=pos_base)
    g = np64(got)
    assert np.array_equal(g, want), f"{int((g != want).sum())} of {g.size} differ"


# ------------------------------------------------------------------ Q prologue
@pytest.mark.parametrize("rows,q_base", [(333, 0), (200, 704)])
def test_q_prologue_bit_exact(rows, q_base):
    inp = Inputs(SEED + 9, rows, q_base + rows)
    d = inp.dev()
    got = B.ga_q_prologue(d["qg"], d["w_q"], d["cos"], d["sin"], q_base=q_base)
    c, s = inp.oracle_tables()
    want, _ = O.prep_queries(inp.np["qg"], inp.np["w_q"], c, s, q_base)
    g = np64(got)
    assert np.array_equal(g, want), f"{int((g != want).sum())} of {g.size} differ"


def test_q_prologue_bit_exact_s8192():
    """The query prologue over the headline configuration's 8192 x 24 rows: every prepared
    value equals the oracle's. About one row in ten has an element near a bf16 rounding
    midpoint and takes the kernel's exact path, so both paths are covered many times."""
    S = 8192
    qg = synth.normal_bf16(SEED + 11, "qg", (S, 24, 512))
    w_q = synth.normal_bf16(SEED + 11, "w_q", (256,), sigma=0.1)
    c, s = B.ga_rope_table_host(S)
    got = B.ga_q_prologue(qg.cuda(), w_q.cuda(), c.cuda(), s.cuda())
    oc, os_ = O.rope_tables(S)
    want, _ = O.prep_queries(np64(qg), np64(w_q), oc, os_, 0)
    g = np64(got)
    assert np.array_equal(g, want), f"{int((g != want).sum())} of {g.size} differ"


@pytest.mark.parametrize("n_tok,k_pos,rows,q_base", [(2048, 0, 333, 0), (333, 777, 200, 704),
                                                    (0, 0, 100, 0), (50, 3, 0, 0),
                                                    (8192, 0, 8192, 0)])
def test_qk_prologue_equals_single_calls(n_tok, k_pos, rows, q_base):
    """Both prologues in one launch: the same bits as ga_k_prologue and ga_q_prologue, with
    the runs of key and query rows dealt over one grid (an empty run, whose output stays
    untouched; a key run shorter than the grid's half-warps; the full S = 8192 pass); the
    oracle fixes the small cases."""
    T = max(k_pos + n_tok, q_base + rows, 1)
    c, s = B.ga_rope_table_host(T)
    cos, sin = c.cuda(), s.cuda()
    w_k = synth.normal_bf16(SEED + 13, "w_k", (256,), sigma=0.1).cuda()
    w_q = synth.normal_bf16(SEED + 13, "w_q", (256,), sigma=0.1).cuda()
    # buffers of at least one row, so that an empty run still passes valid pointers
    k = synth.normal_bf16(SEED + 13, "k", (max(n_tok, 1), 2, 256)).cuda()
    qg = synth.normal_bf16(SEED + 13, "qg", (max(rows, 1), 24, 512)).cuda()
    kp = torch.full_like(k, 7.0)
    qp = torch.full((max(rows, 1), 24, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    st = B.lib().ga_qk_prologue(k.data_ptr(), w_k.data_ptr(), n_tok, k_pos, kp.data_ptr(),
                                qg.data_ptr(), w_q.data_ptr(), rows, q_base, qp.data_ptr(),
                                cos.data_ptr(), sin.data_ptr(), T, B._stream())
    assert st == 0
    torch.cuda.synchronize()
    assert B.ga_device_status() == 0
    if n_tok:
        want_k = B.ga_k_prologue(k, w_k, cos, sin, pos_base=k_pos)
        assert torch.equal(kp.view(torch.int16), want_k.view(torch.int16))
    else:
        assert bool((kp == 7.0).all())
    if rows:
        want_q = B.ga_q_prologue(qg, w_q, cos, sin, q_base=q_base)
        assert torch.equal(qp.view(torch.int16), want_q.view(torch.int16))
    else:
        assert bool((qp == 7.0).all())
    if T <= 4096:
        oc, os_ = O.rope_tables(T)
        if n_tok:
            wk = O.prep_keys(np64(k.cpu()), np64(w_k.cpu()), oc, os_, pos0=k_pos)
            assert np.array_equal(np64(kp), wk)
        if rows:
            wq, _ = O.prep_queries(np64(qg.cpu()), np64(w_q.cpu()), oc, os_, q_base)
            assert np.array_equal(np64(qp), wq)


def test_qk_prologue_binding():
    """The binding's form allocates both outputs and returns them."""
    T = 640
    c, s = B.ga_rope_table_host(T)
    k = synth.normal_bf16(SEED + 14, "k", (T, 2, 256)).cuda()
    qg = synth.normal_bf16(SEED + 14, "qg", (128, 24, 512)).cuda()
    w = synth.normal_bf16(SEED + 14, "w_q", (256,), sigma=0.1).cuda()
    kp, qp = B.ga_qk_prologue(k, w, qg, w, c.cuda(), s.cuda(), q_base=512)
    assert kp.shape == k.shape and qp.shape == (128, 24, 256)
    assert torch.equal(kp.view(torch.int16),
                       B.ga_k_prologue(k, w, c.cuda(), s.cuda()).view(torch.int16))
    assert torch.equal(qp.view(torch.int16),
                       B.ga_q_prologue(qg, w, c.cuda(), s.cuda(), q_base=512).view(torch.int16))


def test_prepared_path_matches_fused_call():
    """ga_q_prologue + ga_attn_prefill_prepared equals ga_attn_prefill bit for bit, with the
    prepared queries in their own buffer and in the output buffer itself."""
    S = 1000
    inp = Inputs(SEED + 10, S, S)
    d = inp.dev()
    full = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    qp = B.ga_q_prologue(d["qg"], d["w_q"], d["cos"], d["sin"])
    sep = B.ga_attn_prefill_prepared(qp, d["qg"], d["k_prep"], d["v"])
    assert torch.equal(sep, full)
    out = torch.empty_like(full)
    B.ga_q_prologue(d["qg"], d["w_q"], d["cos"], d["sin"], q_prep=out.view(S, 24, 256))
    B.ga_attn_prefill_prepared(out, d["qg"], d["k_prep"], d["v"], out=out)
    assert torch.equal(out, full)


# ------------------------------------------------------------------ tiny and S=2048
def test_prefill_tiny_s64_all_heads():
    inp = Inputs(SEED + 1, 64, 64)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 64)
    inp.ref(0, 64, "causal").check(got, what="S=64 causal")
    for mode in ("R2", "F64"):   # information: the other readings of the rounding point
        print(f"[info] S=64 GPU vs {mode}:", compare(got, _oracle_prefill(inp, 0, 64, True, mode=mode)))


def test_prefill_causal_s2048_all_heads():
    inp = Inputs(SEED + 2, 2048, 2048)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 2048)
    inp.ref(0, 2048, "causal").check(got, what="S=2048 causal, all rows and heads")


def test_prefill_bidirectional_s2048():
    inp = Inputs(SEED + 2, 2048, 2048)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 2048,
                            causal=False)
    heads = [0, 7, 11, 12, 18, 23]
    inp.ref(0, 2048, "bidirectional", heads=heads).check(
        got, what="S=2048 bidirectional (6 heads, all rows)")
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    inp.ref(0, 2048, "bidirectional", rows=rows).check(
        got[torch.as_tensor(rows)], what="S=2048 bidirectional (all heads, 6 rows)")


# ------------------------------------------------------------------ ragged and windows
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_ragged_rows_and_keys(causal):
    S = 333
    inp = Inputs(SEED + 3, S, S)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                            causal=causal)
    inp.ref(0, S, "causal" if causal else "bidirectional").check(got, what=f"S=333 causal={causal}")


@pytest.mark.parametrize("q_base", [64, 128, 192])
def test_prefix_window_ragged(q_base):
    S = 333
    inp = Inputs(SEED + 3, S, S)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"][q_base:], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                            q_base, S)
    inp.ref(q_base, S, "causal", qg=inp.np["qg"][q_base:]).check(got, what=f"window q_base={q_base}")


def test_windows_bit_identical_to_full_pass():
    """system1-omni PR #202 §Test Plan: prefix windows at q_base 64/128/1,024 match the
    full pass bit for bit."""
    S = 1280
    inp = Inputs(SEED + 4, S, S)
    d = inp.dev()
    full = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    for qb in (64, 128, 1024):
        win = B.ga_attn_prefill(d["qg"][qb:], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                                qb, S)
        assert torch.equal(win, full[qb:]), f"q_base={qb}"
    # a window over a prefix of the keys (T < S) equals the full pass of that prefix
    T = 640
    part = B.ga_attn_prefill(d["qg"][512:640], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                             512, T)
    assert torch.equal(part, full[512:640])


# ------------------------------------------------------------------ edge cases
def test_single_key_and_single_row():
    inp = Inputs(SEED + 5, 1, 1)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 1)
    g = inp.np["qg"][0, :, 256:]
    v = inp.np["v"][0]
    want = np.concatenate([O.bf16(v[h // 12] * O.bf16(1 / (1 + np.exp(-g[h])))) for h in range(24)])
    assert np.array_equal(np64(got)[0], want)


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("q_base", [0, 4096])
def test_gate_every_bf16_value(pairs, q_base):
    """Every bf16 gate value but NaN (one per output element across 11 rows) with V = 1, so
    that o = 1 and out = bf16(sigmoid(g)) itself: the device's sigmoid table, bit for bit
    against the oracle, including +-inf, subnormal gates and the gates whose sigmoid is a
    bf16 subnormal. Both forms of the kernel: CTA pairs (their gate tiles through the
    staging buffer) and single CTAs (through the ring), for the rows at the start of the
    sequence and as a window at q_base 4096 over 4,107 keys."""
    bits = np.arange(65536, dtype=np.uint32)
    is_nan = (((bits >> 7) & 0xFF) == 0xFF) & ((bits & 0x7F) != 0)
    vals = (bits[~is_nan] << 16).view(np.float32).astype(np.float64)
    rows = -(-vals.size // 6144)
    T = q_base + rows
    inp = Inputs(SEED + 11, rows, T)
    g = np.zeros(rows * 6144)
    g[:vals.size] = vals
    qg = inp.cpu["qg"].clone()
    qg[:, :, 256:] = torch.from_numpy(g.reshape(rows, 24, 256)).to(torch.bfloat16)
    inp.cpu["qg"], inp.np["qg"] = qg, np64(qg)
    inp.cpu["v"] = torch.ones_like(inp.cpu["v"])
    inp.np["v"] = np64(inp.cpu["v"])
    d = inp.dev()
    prev = B.ga_debug_set_cta_pairs(2 if pairs else 0)
    try:
        got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                                q_base, T)
        torch.cuda.synchronize()
    finally:
        B.ga_debug_set_cta_pairs(prev)
    # with every value 1, o = bf16(O / l) = 1 for any weights: the output is the gate's
    # rounded sigmoid, which the oracle's full pass confirms on the small case
    want = O.sigmoid_gate(g).reshape(rows, 24 * 256)
    if q_base == 0:
        assert np.array_equal(inp.ref(0, rows, "causal").out.reshape(-1), want.reshape(-1))
    g_np = np64(got)
    diff = np.flatnonzero(g_np.reshape(-1)[:vals.size] != want.reshape(-1)[:vals.size])
    assert diff.size == 0, f"{diff.size} gates differ, e.g. g={g[diff[:5]]}"


def test_row_stats_and_hidden_free_causal():
    inp = Inputs(SEED + 6, 256, 256)
    d = inp.dev()
    stats = torch.full((24, 256, 2), float("nan"), device="cuda")
    B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 256,
                      row_stats=stats)
    st = stats.cpu().numpy()
    # M is ceil(max t) when first set and the row's largest weight is at least 2^-1
    assert np.all(np.isfinite(st)) and np.all(st[..., 1] >= 0.5)
    assert np.all(st[..., 0] == np.round(st[..., 0]))


# ------------------------------------------------------------------ S = 8192
def test_prefill_s8192_full_and_chunks():
    """Long causal prefill at S=8192: the full pass against the oracle on sampled rows,
    and two 4096-row chunks (q_base 0, then 4096 over the accumulated keys) bit-identical
    to the full pass's rows."""
    S = 8192
    inp = Inputs(SEED + 8, S, S)
    d = inp.dev()
    full = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    c1 = B.ga_attn_prefill(d["qg"][:4096], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                           0, 4096)
    c2 = B.ga_attn_prefill(d["qg"][4096:], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                           4096, S)
    assert torch.equal(c1, full[:4096])
    assert torch.equal(c2, full[4096:])
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 4096, 4097, 8063, 8064, 8191],
                                     rng.integers(0, S, 22)]))
    inp.ref(0, S, "causal", rows=rows).check(full[torch.as_tensor(rows)],
                                              what=f"S=8192 causal, {len(rows)} sampled rows")
    r2 = rows[rows >= 4096] - 4096
    inp.ref(4096, S, "causal", rows=r2, qg=inp.np["qg"][4096:]).check(
        c2[torch.as_tensor(r2)], what=f"S=8192 chunk q_base=4096, {len(r2)} sampled rows")


# ------------------------------------------------------------------ negative controls
def test_negative_control_kv_swap_fails():
    """pegainfer PR #1151 §Validation: exchanging the two KV heads must fail the gate."""
    inp = Inputs(SEED + 1, 64, 64)
    d = inp.dev()
    swapped = d["k_prep"].flip(1).contiguous()
    got = B.ga_attn_prefill(d["qg"], swapped, d["v"], d["w_q"], d["cos"], d["sin"], 0, 64)
    with pytest.raises(AssertionError):
        inp.ref(0, 64, "causal").check(got, what="KV heads swapped (must fail)")
