"""CPU oracle for gated grouped-query attention (test infrastructure only).

This is the plain, slow, obviously-correct statement of what the GB300 library
computes. It is test infrastructure: only the tests, the package smoke check and the
benchmark's CPU-baseline leg use it. It shares no code with the CUDA path (it imports
only numpy) and everything is float64 except at the rounding points listed below.

Sources (the pull-request pages this method is read from):
  [QSA]    pegainfer PR #1151, "feat(qwen4): add the QSA sparse-attention kernel and
           its golden" -- §Semantics; §What changed; §Validation; the commit message
           that adds the attention reader ("Rounding is reproduced at every point the
           reference rounds ..."); review item F4 on the frequency table.
  [WIDE]   system1-omni PR #202, "cuda: widen the attention query tile on sm_89 and
           sm_120" -- §Scope (windows and bidirectional pass), first review §Kernel
           change (online-softmax recurrence, masked lanes), §Dispatch/guard.
  [LONG]   TensorFold PR #1080, "qwen CUDA: long-prompt prefill 5.4x faster" --
           the attn_partial commit (split chunks, partials and their combine).

Geometry (QSA, the commit replacing the proxy geometry): 24 query heads, 2 KV heads,
group 12 (query head h reads KV head h // 12), head_dim 256, RoPE on dims 0..63,
rms_norm_eps 1e-6, RoPE base 1e7.

Rounding points (QSA §Semantics and the attention-reader commit): the norms are cast
to bf16 once; cos/sin are bf16 and the rotation rounds in bf16; the score is the bf16
rounding of q.k before the exact 1/16 scale; the softmax weight is rounded to bf16
before the context reduction; the sigmoid of the gate rounds to bf16 before the final
product, which rounds again. All roundings are round-to-nearest-even.

Softmax rounding point. The pages describe two placements of "weights rounded to bf16
before the context reduction": QSA's materialised kernel normalises first and rounds
w = bf16(softmax(s)) (mode "R2"); the flash recurrence of [WIDE] rounds the
unnormalised exponential P before P.V and divides by the running sum afterwards. Mode
"R1" (primary) states the latter independently of any tile schedule:
    w_hat_ij = e^{s_ij} rounded to bf16's 8-bit significand (exponent unbounded),
    L_i = sum_j w_hat_ij over visible j,   o_i = bf16( sum_j w_hat_ij v_j / L_i ).
Mode "F64" rounds nothing after the inputs (tables unrounded too).
"""
from __future__ import annotations

import math

import numpy as np

N_Q_HEADS = 24
N_KV_HEADS = 2
GROUP = N_Q_HEADS // N_KV_HEADS
HEAD_DIM = 256
ROT_DIMS = 64
HALF_ROT = ROT_DIMS // 2
EPS = 1e-6
ROPE_BASE = 1e7
MODES = ("R1", "R2", "F64")


# ----------------------------------------------------------------------------------
# bf16 rounding
# ----------------------------------------------------------------------------------
def bf16(x):
    """Round float64 values to the nearest bfloat16 value (ties to even), as float64.

    bfloat16 keeps 8 significant bits and float32's exponent range: normal values
    down to 2^-126, subnormals in steps of 2^-133, overflow to +-inf past the largest
    finite value (2 - 2^-7) * 2^127.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                 # quantum 2^(e-8), floored at 2^-133
    q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    q = np.where(np.abs(q) >= 2.0 ** 128, np.copysign(np.inf, x), q)
    return q


def bf16_sig(x):
    """Round to bf16's 8-bit significand with an unbounded exponent (R1's w_hat)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def ulp_bf16(x):
    """Spacing of bf16 values at |x|: 2^(floor(log2|x|) - 7); 2^-133 below 2^-126."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    m, e = np.frexp(np.where(x > 0, x, 1.0))
    u = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    return np.where(x > 0, u, 2.0 ** -133)


def within_tolerance(got, want, n_ulp=2.0, atol=1e-5):
    """Element-wise check |got - want| <= n_ulp * ulp(want) + atol (bool array)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return np.abs(got - want) <= n_ulp * ulp_bf16(want) + atol


# ----------------------------------------------------------------------------------
# RoPE table, (1+w) RMSNorm, partial RoPE
# ----------------------------------------------------------------------------------
def rope_tables(n_pos, rounded=True, base=ROPE_BASE, rot_dims=ROT_DIMS):
    """cos and sin tables [n_pos, rot_dims/2].

    Angle of position p and pair i: p * base^(-2i/rot_dims), computed in float64 and
    (when rounded) rounded once to bf16. [QSA] review F4: the kernel side builds the
    table with a double pow and rounds it once; both kernels read one shared table, so
    no trigonometry runs on the device ([QSA] §What changed).
    """
    # The C library's math (correctly rounded pow; cos and sin to within an ulp), one
    # element at a time: numpy's vectorised pow is not correctly rounded for every i.
    inv_freq = np.array([math.pow(base, -(2.0 * i) / rot_dims) for i in range(rot_dims // 2)])
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.frompyfunc(math.cos, 1, 1)(ang).astype(np.float64)
    s = np.frompyfunc(math.sin, 1, 1)(ang).astype(np.float64)
    if rounded:
        return bf16(c), bf16(s)
    return c, s


def rms_norm_1pw(x, w, eps=EPS, rounded=True):
    """(1+w) RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * (1 + w).

    [QSA] §Semantics ("(1+w) RMSNorm on q and k at rms_norm_eps") and the
    attention-reader commit ("the norms cast once"): float64, one bf16 rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = (x * r) * (1.0 + np.asarray(w, dtype=np.float64))
    return bf16(y) if rounded else y


def rope_partial(x, cos_rows, sin_rows, rounded=True):
    """Rotate-half RoPE on dims 0..63 of the last axis; dims 64..255 pass through.

    Pair i < 32 is (x_i, x_{i+32}) rotated by angle i. [QSA] §Semantics ("64-of-256
    partial RoPE from the shared table") and the attention-reader commit ("cos/sin are
    cast to bf16 and rotate in bf16"): each product rounds to bf16, then the sum.
    cos_rows/sin_rows broadcast against x[..., :32].
    """
    x = np.asarray(x, dtype=np.float64)
    a = x[..., :HALF_ROT]
    b = x[..., HALF_ROT:ROT_DIMS]
    y = x.copy()
    if rounded:
        y[..., :HALF_ROT] = bf16(bf16(a * cos_rows) - bf16(b * sin_rows))
        y[..., HALF_ROT:ROT_DIMS] = bf16(bf16(b * cos_rows) + bf16(a * sin_rows))
    else:
        y[..., :HALF_ROT] = a * cos_rows - b * sin_rows
        y[..., HALF_ROT:ROT_DIMS] = b * cos_rows + a * sin_rows
    return y


def prep_keys(k_raw, w_k, cos, sin, pos0=0, mode="R1"):
    """Prepared keys [T, 2, 256]: (1+w_k) norm, then RoPE at position pos0 + t.

    [QSA] §What changed: one key pass norms and rotates every token's two key heads
    once, because all twelve query heads of a KV head read the same prepared key.
    """
    rounded = mode != "F64"
    k = np.asarray(k_raw, dtype=np.float64)
    T = k.shape[0]
    pos = pos0 + np.arange(T)
    kn = rms_norm_1pw(k, w_k, rounded=rounded)
    return rope_partial(kn, cos[pos][:, None, :], sin[pos][:, None, :], rounded=rounded)


def prep_queries(qg, w_q, cos, sin, q_base, mode="R1", rows=None):
    """Split the fused rows, norm and rotate q. Returns (q_hat, gate), [n, 24, 256].

    [QSA] §Semantics: "the q|gate split of the fused q_proj row"; per head the first
    256 values are q and the last 256 the gate. Query row r sits at position q_base + r.
    rows selects a subset of the window's rows (default: all).
    """
    rounded = mode != "F64"
    qg = np.asarray(qg, dtype=np.float64)
    if rows is None:
        rows = np.arange(qg.shape[0])
    rows = np.asarray(rows)
    q = qg[rows, :, :HEAD_DIM]
    g = qg[rows, :, HEAD_DIM:]
    pos = q_base + rows
    qn = rms_norm_1pw(q, w_q, rounded=rounded)
    qh = rope_partial(qn, cos[pos][:, None, :], sin[pos][:, None, :], rounded=rounded)
    return qh, g


# ----------------------------------------------------------------------------------
# Visibility
# ----------------------------------------------------------------------------------
def visibility(kind, rows, T, q_base=0, mask=None):
    """bool [len(rows), T]: which keys each query row sees.

    causal:        key j <= q_base + r  (a prefix window when q_base > 0) [WIDE] §Scope
    bidirectional: every key j < T (q_base must be 0)                     [WIDE] §Scope
    mask:          mask[r, j] != 0, the stored mask as given, not ANDed with
                   causality by the kernel                                [QSA] §Semantics
    """
    rows = np.asarray(rows)
    j = np.arange(T)
    if kind == "causal":
        return j[None, :] <= (q_base + rows)[:, None]
    if kind == "bidirectional":
        return np.ones((len(rows), T), dtype=bool)
    if kind == "mask":
        return np.asarray(mask)[rows, :T] != 0
    raise ValueError(kind)


# ----------------------------------------------------------------------------------
# Selection mask: the indexer's top-k blocks AND causality
# ----------------------------------------------------------------------------------
# [QSA], the commit moving the oracle to the real geometry: an indexer budget of 2048
# tokens is 512 blocks, so a block holds 4 consecutive keys; its golden review: budget
# 16 -> block_topk 4.
BLOCK_TOKENS = 4


def block_topk_for_budget(budget):
    """Blocks a row keeps for a token budget: budget / BLOCK_TOKENS (2048 -> 512, 16 -> 4)."""
    budget = int(budget)
    if budget < BLOCK_TOKENS or budget % BLOCK_TOKENS:
        raise ValueError("the budget is a positive multiple of the block size")
    return budget // BLOCK_TOKENS


def select_blocks_mask(block_scores, q_base, T, block_topk):
    """uint8 [rows, T], 1 = visible: the mask the stored-mask pass reads, built from the
    indexer's per-block scores ([QSA] the attention-reader commit: the mask is the
    indexer's selection AND causality; the golden's effective mask is the same AND).

    block_scores [rows, >= ceil(T / 4)]: row r (position p = q_base + r) scores block b,
    the keys 4b .. 4b + 3. The row's candidates are the blocks holding a key j <= p, that
    is b = 0 .. p // 4. It keeps the block_topk candidates with the highest scores, a tie
    going to the lower block index (every candidate when there are fewer), and sees key j
    iff j <= p and block j // 4 is kept. Scores may be +-inf, never NaN; -0 equals +0."""
    s = np.asarray(block_scores, np.float64)
    rows = s.shape[0]
    nb = -(-T // BLOCK_TOKENS)
    assert block_topk >= 1 and q_base >= 0 and q_base + rows <= T
    assert not np.isnan(s[:, :nb]).any(), "scores must not be NaN"
    j = np.arange(T)
    out = np.zeros((rows, T), np.uint8)
    for r in range(rows):
        p = q_base + r
        nc = min(nb, p // BLOCK_TOKENS + 1)
        cand = np.arange(nc)
        order = np.lexsort((cand, -s[r, :nc]))      # score descending, then index ascending
        kept = np.zeros(nb, dtype=bool)
        kept[order[:block_topk]] = True
        out[r] = (j <= p) & kept[j // BLOCK_TOKENS]
    return out


# ----------------------------------------------------------------------------------
# The attention core
# ----------------------------------------------------------------------------------
def sigmoid_gate(g, mode="R1"):
    """sigmoid(g) = 1 / (1 + e^{-g}); rounded to bf16 except in F64 ([QSA] §Semantics).
    For g below about -709, e^{-g} overflows to inf and the quotient is the exact limit 0."""
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-np.asarray(g, dtype=np.float64)))
    return s if mode == "F64" else bf16(s)


def scores(q_hat, k_hat, mode="R1"):
    """s_ij = bf16(q_i . k_j) * 2^-4: the bf16 rounding of the dot product, then the exact
    1/sqrt(256) ([QSA] attention-reader commit: "the score is the bf16 GEMM result rounded
    before the exact 1/16 scale"). The dot product is formed in float64 (exact for these
    bf16 inputs up to float64 rounding of the running sum)."""
    dot = q_hat @ k_hat.T
    return dot / 16.0 if mode == "F64" else bf16(dot) / 16.0


def attend_scores(s, gate, v, vis, mode="R1", want_weights=False):
    """Softmax over the visible scores, P.V and the gate for one query head.

    s: [n, T] scores; gate: [n, 256]; v: [T, 256]; vis: bool [n, T].
    Returns (out [n, 256], weights [n, T] or None, hidden bool [n]). A row with no visible
    key outputs zeros (the pages leave it outside the contract; it is flagged in `hidden`).
    """
    hidden = ~vis.any(axis=1)
    weights = None
    if mode == "R1":
        w_hat = np.where(vis, bf16_sig(np.exp(np.where(vis, s, 0.0))), 0.0)
        L = w_hat.sum(axis=1, keepdims=True)
        Ls = np.where(L > 0, L, 1.0)
        o = bf16((w_hat @ v) / Ls)
        if want_weights:
            weights = bf16(w_hat / Ls)
    else:
        m = np.max(np.where(vis, s, -np.inf), axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(vis, np.exp(np.where(vis, s - m, 0.0)), 0.0)
        z = e.sum(axis=1, keepdims=True)
        w = e / np.where(z > 0, z, 1.0)
        if mode == "R2":
            w = bf16(w)
            o = bf16(w @ v)
        else:
            o = w @ v
        if want_weights:
            weights = w
    sig = sigmoid_gate(gate, mode)
    out = o * sig if mode == "F64" else bf16(o * sig)
    out = np.where(hidden[:, None], 0.0, out)
    return out, weights, hidden


def attend_head(q_hat, gate, k_hat, v, vis, mode="R1", want_weights=False):
    """One query head over its KV head: q_hat, gate [n, 256]; k_hat, v [T, 256]; vis [n, T]."""
    return attend_scores(scores(q_hat, k_hat, mode), gate, v, vis, mode, want_weights)


def attention(q_hat, gate, k_hat, v, vis, mode="R1", heads=None, want_weights=False):
    """All (or the listed) query heads.

    q_hat, gate [n, 24, 256]; k_hat, v [T, 2, 256]; vis [n, T].
    Returns out [n, 24*256] (head-major columns h*256 + d, zeros for heads not listed),
    weights [24, n, T] (or None), hidden [n].
    """
    n = q_hat.shape[0]
    T = k_hat.shape[0]
    heads = range(N_Q_HEADS) if heads is None else heads
    out = np.zeros((n, N_Q_HEADS * HEAD_DIM))
    weights = np.zeros((N_Q_HEADS, n, T)) if want_weights else None
    v = np.asarray(v, dtype=np.float64)
    hidden = ~vis.any(axis=1)
    for h in heads:
        kv = h // GROUP                       # GQA: query head h reads KV head h // 12
        o, w, _ = attend_head(q_hat[:, h], gate[:, h], k_hat[:, kv], v[:, kv], vis,
                              mode, want_weights)
        out[:, h * HEAD_DIM:(h + 1) * HEAD_DIM] = o
        if want_weights:
            weights[h] = w
    return out, weights, hidden


# ----------------------------------------------------------------------------------
# The three entry points, stated whole
# ----------------------------------------------------------------------------------
def prefill(qg, k_prep, v, w_q, cos, sin, q_base, T, causal=True, mode="R1",
            rows=None, heads=None):
    """Causal (or prefix-window) / bidirectional gated GQA over prepared keys.

    qg [rows_total, 24, 512] holds the window's rows at positions q_base + r; k_prep and
    v hold keys 0 .. T-1. rows/heads select a sample of the outputs.
    [WIDE] §Scope: full pass (causal or bidirectional) and prefix windows at q_base.
    """
    if rows is None:
        rows = np.arange(np.asarray(qg).shape[0])
    q_hat, gate = prep_queries(qg, w_q, cos, sin, q_base, mode, rows)
    vis = visibility("causal" if causal else "bidirectional", rows, T, q_base)
    out, _, _ = attention(q_hat, gate, np.asarray(k_prep, np.float64)[:T], v[:T], vis,
                          mode, heads)
    return out


def masked(qg, k_prep, v, w_q, cos, sin, q_base, T, mask, mode="R1", rows=None,
           heads=None, want_weights=False):
    """Stored-mask attention ([QSA] §Semantics): mask row r is position q_base + r."""
    if rows is None:
        rows = np.arange(np.asarray(qg).shape[0])
    q_hat, gate = prep_queries(qg, w_q, cos, sin, q_base, mode, rows)
    vis = visibility("mask", rows, T, q_base, mask)
    return attention(q_hat, gate, np.asarray(k_prep, np.float64)[:T], v[:T], vis, mode,
                     heads, want_weights)


def verify(qg_seq, k_cache, v_cache, seq_len, w_q, cos, sin, mode="R1", rows=None,
           heads=None):
    """Few-row verify windows: sequence b's row r sits at position L_b + r and sees
    prepared cache keys 0 .. L_b + r ([LONG], the attn_partial commit: split chunks
    and their combine compute exactly this causal attention).

    qg_seq [n_seq, R, 24, 512]; k_cache, v_cache [n_seq, cap, 2, 256] (prepared keys).
    Returns out [n_seq, R, 24*256].
    """
    qg_seq = np.asarray(qg_seq)
    n_seq, R = qg_seq.shape[0], qg_seq.shape[1]
    outs = []
    for b in range(n_seq):
        L = int(seq_len[b])
        T = L + R
        outs.append(prefill(qg_seq[b], k_cache[b], v_cache[b], w_q, cos, sin, L, T,
                            True, mode, rows, heads))
    return np.stack(outs)


E4M3_MAX = 448.0


def e4m3(x):
    """Round float64 values to the OCP FP8 E4M3 grid (sign, 4 exponent bits with bias 7,
    3 mantissa bits, subnormals down to 2^-9, no infinities), nearest with ties to even,
    saturating to +-448 (the 'satfinite' conversion)."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                        # below 2^-6 the grid is subnormal, 2^-9 apart
    quantum = np.exp2(e - 3.0)
    q = np.round(a / quantum) * quantum            # np.round: ties to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(a > 0, np.sign(x) * q, x * 0.0)


def fp32(x):
    """Round float64 values to float32 (nearest, ties to even), as float64."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def quantize_e4m3_rows(x):
    """e4m3 cache rows with one fp32 scale each (TensorFold PR #1080, "qwen CUDA: long-prompt
    prefill 5.4x faster", the prompt-chain commit: e4m3 cache rows with an fp32 scale each,
    widened to bf16 in the slot; the rope-kernel commit computes the e4m3 scales by block
    reductions). Over the last axis (one row): sc = fp32(max|x| / 448), q = e4m3(fp32(x / sc)),
    both divisions and roundings as fp32 arithmetic would do them; a zero row has sc = 0 and
    q = 0. Returns (q as float64 values on the e4m3 grid, sc)."""
    x = np.asarray(x, np.float64)
    a = np.max(np.abs(x), axis=-1, keepdims=True)
    sc = fp32(a.astype(np.float32) / np.float32(E4M3_MAX))
    safe = np.where(sc > 0, sc, 1.0).astype(np.float32)
    ratio = (x.astype(np.float32) / safe).astype(np.float64)
    q = np.where(sc > 0, e4m3(ratio), 0.0)
    return q, sc[..., 0]


def dequantize_e4m3_rows(q, sc):
    """The widened bf16 row: bf16(fp32(q * sc)) per element."""
    prod = (np.asarray(q, np.float64).astype(np.float32) *
            np.asarray(sc, np.float64)[..., None].astype(np.float32)).astype(np.float64)
    return bf16(prod)


def gather_pages(pool, table_row, n_tok, page_size):
    """A sequence's cache rows 0 .. n_tok-1 from a page pool: position t lives on page
    table_row[t // page_size], slot t % page_size. pool [n_pages, page_size, ...].
    (Paged caches are named as the next step after the contiguous key array in [QSA]
    §Summary and §Limits; the layout is this plain reading of a page table.)"""
    pool = np.asarray(pool)
    rows = []
    for t in range(n_tok):
        rows.append(pool[int(table_row[t // page_size]), t % page_size])
    if not rows:
        return np.zeros((0,) + pool.shape[2:], dtype=pool.dtype)
    return np.stack(rows)


def verify_paged(qg_seq, k_pages, v_pages, page_table, page_size, seq_len, w_q, cos, sin,
                 mode="R1", rows=None, heads=None):
    """verify() over paged caches: each sequence's prepared keys and values are gathered
    from the page pools through its page-table row, then attended exactly as in verify().
    Decode is the same with one row per sequence."""
    qg_seq = np.asarray(qg_seq)
    R = qg_seq.shape[1]
    outs = []
    for b in range(qg_seq.shape[0]):
        L = int(seq_len[b])
        kc = gather_pages(k_pages, page_table[b], L + R, page_size)
        vc = gather_pages(v_pages, page_table[b], L + R, page_size)
        outs.append(prefill(qg_seq[b], kc, vc, w_q, cos, sin, L, L + R, True, mode, rows,
                            heads))
    return np.stack(outs)

