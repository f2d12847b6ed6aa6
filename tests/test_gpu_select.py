"""GPU parity of the selection-mask producer: every mask byte equal to the oracle's (integer
work, so bit-exact), at the full 8192 x 8192 size with a budget of 2048 tokens, on tie-heavy,
signed-zero and infinite scores, ragged T, windows at q_base > 0, strided score rows, and
through the stored-mask attention it feeds."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, np64
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


def _check(scores, T, q_base, k, ld_pad=0, what=""):
    """scores: float32 CPU tensor [rows, >= ceil(T/4)]; the GPU mask against the oracle's,
    with the columns past T left as they were (7)."""
    rows = scores.shape[0]
    ld = (T + 15) // 16 * 16 + ld_pad
    mask = torch.full((rows, ld), 7, dtype=torch.uint8, device="cuda")
    B.ga_select_mask(scores.cuda(), T, k, q_base=q_base, mask=mask)
    got = mask.cpu().numpy()
    want = O.select_blocks_mask(scores.double().numpy(), q_base, T, k)
    bad = np.argwhere(got[:, :T] != want)
    assert bad.size == 0, (what, bad[:5])
    assert np.all(got[:, T:] == 7), what
    return got[:, :T]


def test_select_full_size_budget_2048():
    """8192 query rows over 8192 keys, 2048 blocks of N(0,1) scores, block_topk 512 (a
    budget of 2048 tokens): the whole mask, byte for byte."""
    T, k = 8192, O.block_topk_for_budget(2048)
    scores = synth.block_scores(SEED + 90, T, T // 4)
    m = _check(scores, T, 0, k, what="8192 x 8192")
    kept = m.sum(1)
    assert kept[-1] == 4 * k and kept[100] == 101       # truncated row / causal row


@pytest.mark.parametrize("T,q_base,k,kind", [
    (1, 0, 1, "normal"), (5, 0, 1, "ties"), (17, 3, 2, "special"), (1203, 5, 37, "ties"),
    (1203, 5, 37, "normal"), (4096, 1000, 1, "normal"), (4096, 0, 1024, "ties"),
    (8192, 8000, 300, "special"), (999, 0, 250, "normal"), (64, 0, 10 ** 6, "normal")])
def test_select_edge_cases(T, q_base, k, kind):
    """Single key, T not a multiple of 4 or 16, windows, k = 1, k >= every row's
    candidates, scores rounded to few values (ties everywhere), and +-0 / +-inf mixed in."""
    rows = T - q_base
    nb = -(-T // 4)
    s = synth.block_scores(SEED + 91 + T + k, rows, nb)
    if kind == "ties":
        s = torch.round(s * 2.0)
    elif kind == "special":
        vals = torch.tensor([-float("inf"), -1.0, -0.0, 0.0, 0.5, 1.0, float("inf")])
        idx = torch.from_numpy(np.random.default_rng(T).integers(0, 7, (rows, nb)))
        s = vals[idx]
    _check(s, T, q_base, k, what=f"T={T} q_base={q_base} k={k} {kind}")


def test_select_strided_scores_and_wide_mask():
    """Score rows with a leading dimension above ceil(T/4) (a column slice of a wider
    array) and a mask wider than T."""
    T, k = 2000, 64
    wide = synth.block_scores(SEED + 92, T, 700)
    scores = wide[:, 100:600]                  # 500 = ceil(2000 / 4) blocks, ld 700
    rows = T
    mask = torch.full((rows, 2048 + 32), 7, dtype=torch.uint8, device="cuda")
    sc = wide.cuda()[:, 100:600]
    B.ga_select_mask(sc, T, k, mask=mask)
    got = mask.cpu().numpy()
    want = O.select_blocks_mask(scores.double().numpy(), 0, T, k)
    assert np.array_equal(got[:, :T], want)
    assert np.all(got[:, T:] == 7)


def test_selected_mask_feeds_masked_attention():
    """Block scores -> ga_select_mask -> ga_attn_masked, against the oracle's selection and
    the oracle's masked attention (sampled heads), at S = 512 with a 64-token budget."""
    from tests.parity import AttnRef
    S, k = 512, O.block_topk_for_budget(64)
    qg, kr, v, w_q, w_k = synth.attention_inputs(SEED + 93, S, S)
    scores = synth.block_scores(SEED + 93, S, S // 4)
    c, s = B.ga_rope_table_host(S)
    c, s = c.cuda(), s.cuda()
    kd = B.ga_k_prologue(kr.cuda(), w_k.cuda(), c, s)
    mask = B.ga_select_mask(scores.cuda(), S, k)
    out, _, hidden = B.ga_attn_masked(qg.cuda(), kd, v.cuda(), w_q.cuda(), c, s, mask)
    torch.cuda.synchronize()
    assert int(hidden.item()) == 0
    want_mask = O.select_blocks_mask(scores.double().numpy(), 0, S, k)
    assert np.array_equal(mask.cpu().numpy()[:, :S], want_mask)
    oc, os_ = O.rope_tables(S)
    kp = O.prep_keys(np64(kr), np64(w_k), oc, os_)
    AttnRef(np64(qg), kp, np64(v), np64(w_q), oc, os_, 0, S, "mask", mask=want_mask,
            heads=[0, 13, 23]).check(out, what="selected mask through ga_attn_masked")


def test_select_windows_equal_full_pass_rows():
    """Windows at several q_base (rows of the same score array) give the full pass's rows
    byte for byte, and the full pass equals the oracle."""
    T, k = 4096, 256
    scores = synth.block_scores(SEED + 94, T, T // 4).cuda()
    full = B.ga_select_mask(scores, T, k)
    for q_base, rows in ((0, 128), (1000, 77), (4095, 1)):
        win = B.ga_select_mask(scores[q_base:q_base + rows], T, k, q_base=q_base)
        assert torch.equal(win, full[q_base:q_base + rows]), q_base
    want = O.select_blocks_mask(scores.cpu().double().numpy(), 0, T, k)
    assert np.array_equal(full.cpu().numpy()[:, :T], want)


def test_select_nan_row_stays_in_its_row():
    """NaN scores are outside the contract: the call still completes, writes only the NaN
    rows' own mask bytes (inside causality), and every other row equals the oracle's."""
    T, k = 2048, 64
    scores = synth.block_scores(SEED + 95, T, T // 4)
    bad = [100, 1500, 2047]
    for r in bad:
        scores[r, ::3] = float("nan")
    mask = torch.full((T, T + 16), 7, dtype=torch.uint8, device="cuda")
    B.ga_select_mask(scores.cuda(), T, k, mask=mask)
    torch.cuda.synchronize()
    got = mask.cpu().numpy()
    assert np.all(got[:, T:] == 7)
    ok = [r for r in range(T) if r not in bad]
    clean = scores.clone()
    clean[bad] = 0.0
    want = O.select_blocks_mask(clean.double().numpy(), 0, T, k)
    assert np.array_equal(got[ok, :T], want[ok])
    causal = np.arange(T)[None, :] <= np.array(bad)[:, None]
    assert np.all(got[bad, :T] <= causal)
