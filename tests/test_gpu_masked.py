"""GPU parity of stored-mask attention (outputs, weights, hidden rows) against the oracle,
and exact cross-checks against the causal and bidirectional entry points."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, Inputs, np64
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


def test_masked_small_with_weights_and_hidden_row():
    """Small masked case: causal window of 16 plus 64 random keys per row (the selection
    recipe scaled down), one fully hidden row, weights requested."""
    S = 256
    inp = Inputs(SEED + 20, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 20, S, window=16, n_random=64)
    mask[77] = 0                                     # a row with no visible key
    out, w, hid = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                                   mask.cuda(), want_weights=True)
    ref = inp.ref(0, S, "mask", mask=mask.numpy(), want_weights=True)
    ref.check(out, w, "masked S=256 out + weights")
    assert int(hid.item()) == int(ref.hidden.sum()) == 1
    assert torch.all(out[77] == 0) and torch.all(w[:, 77] == 0)
    vis = mask.numpy() != 0
    assert np.all(np64(w)[:, ~vis] == 0)            # hidden keys carry exactly zero weight


def test_masked_ragged_and_window():
    S, qb = 333, 64
    inp = Inputs(SEED + 21, S, S)
    d = inp.dev()
    full_mask = synth.selection_mask(SEED + 21, S, window=32, n_random=40)
    m = full_mask[qb:].contiguous()
    padded = torch.zeros(S - qb, 336, dtype=torch.uint8)   # leading dimension 336 (16-aligned)
    padded[:, :S] = m
    out, w, hid = B.ga_attn_masked(d["qg"][qb:], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                   d["sin"], padded.cuda()[:, :S], q_base=qb, T=S,
                                   want_weights=True)
    ref = inp.ref(qb, S, "mask", mask=m.numpy(), qg=inp.np["qg"][qb:], want_weights=True)
    ref.check(out, w, "masked ragged window out + weights")


def test_masked_equals_causal_and_bidirectional_exactly():
    S = 640
    inp = Inputs(SEED + 22, S, S)
    d = inp.dev()
    tril = torch.tril(torch.ones(S, S, dtype=torch.uint8)).cuda()
    m_out, _, _ = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], tril)
    c_out = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    assert torch.equal(m_out, c_out)
    ones = torch.ones(S, S, dtype=torch.uint8).cuda()
    m_out, _, _ = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], ones)
    b_out = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                              causal=False)
    assert torch.equal(m_out, b_out)


def test_masked_padded_leading_dimension():
    S = 200
    inp = Inputs(SEED + 23, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 23, S, window=8, n_random=30)
    wide = torch.zeros(S, 256, dtype=torch.uint8)
    wide[:, :S] = mask
    wide[:, S:] = 1                                   # padding columns must be ignored
    out, _, _ = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                                 wide.cuda()[:, :S], T=S)
    inp.ref(0, S, "mask", mask=mask.numpy()).check(out, what="masked, ld_mask 256 > T")


def test_masked_s8192_selection_sampled():
    """Sparse-selection masked attention at the 8192 cap: each row sees its causal window
    of 128 keys plus 1024 random earlier keys. Outputs on sampled rows, and weights on the
    last 128-row window."""
    S = 8192
    inp = Inputs(SEED + 24, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 24, S)
    mcu = mask.cuda()
    out, _, hid = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mcu)
    assert int(hid.item()) == 0
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 1151, 1152, 4096, 8191], rng.integers(0, S, 18)]))
    inp.ref(0, S, "mask", rows=rows, mask=mask.numpy()).check(
        out[torch.as_tensor(rows)], what=f"masked S=8192, {len(rows)} rows")
    qb = S - 128
    w_out, w, _ = B.ga_attn_masked(d["qg"][qb:], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                   d["sin"], mcu[qb:], q_base=qb, want_weights=True)
    assert torch.equal(w_out, out[qb:])
    heads = [0, 13]
    ref = inp.ref(qb, S, "mask", mask=mask.numpy()[qb:], qg=inp.np["qg"][qb:], heads=heads,
                  want_weights=True)
    ref.check(w_out, w, "masked S=8192 last window, heads 0/13, out + weights")
    sums = np64(w[heads]).sum(axis=2)
    assert np.all(np.abs(sums - 1) <= 2e-3)


def test_negative_control_causal_for_sparse_mask_fails():
    """pegainfer PR #1151 §Validation: plain causality in place of the stored mask fails."""
    S = 256
    inp = Inputs(SEED + 20, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 20, S, window=16, n_random=64)
    c_out = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    with pytest.raises(AssertionError):
        inp.ref(0, S, "mask", mask=mask.numpy()).check(c_out, what="causal for sparse (must fail)")


def test_masked_prepared_equals_masked_call():
    """ga_q_prologue then ga_attn_masked_prepared gives ga_attn_masked's bits (outputs,
    weights and hidden rows), on a window with a hidden row."""
    S, qb = 384, 128
    inp = Inputs(SEED + 25, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 25, S, window=16, n_random=48)[qb:].contiguous()
    mask[5] = 0
    mcu = mask.cuda()
    qg = d["qg"][qb:]
    ref = B.ga_attn_masked(qg, d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mcu, q_base=qb,
                           want_weights=True)
    q_prep = B.ga_q_prologue(qg, d["w_q"], d["cos"], d["sin"], q_base=qb)
    got = B.ga_attn_masked_prepared(q_prep, qg, d["k_prep"], d["v"], mcu, q_base=qb,
                                    want_weights=True)
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert int(got[2].item()) == int(ref[2].item()) == 1
