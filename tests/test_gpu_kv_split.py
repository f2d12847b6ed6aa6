"""The KV-head split (one GPU per KV head and its 12 query heads, no exchange): the two
groups' calls together give the full call's bits, each writes only its own columns, and
the row windows of a split plan reproduce the full pass too."""
import torch
import pytest

from tests.parity import SEED, Inputs
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod
from verify_gated_gqa_gb300 import shard
from verify_gated_gqa_gb300 import synth

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1   # a NaN no output takes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.lib()
    yield
    assert B.ga_device_status() == 0


def _filled(shape, dev="cuda"):
    return torch.full(shape, SENTINEL, dtype=torch.int16, device=dev).view(torch.bfloat16)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_groups_equal_full_call(causal):
    S = 1000
    inp = Inputs(SEED + 60, S, S)
    d = inp.dev()
    full_stats = torch.zeros(24, S, 2, device="cuda")
    full = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                             causal=causal, row_stats=full_stats)
    out = _filled((S, 6144))
    stats = torch.full((24, S, 2), -7.0, device="cuda")
    B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                      causal=causal, out=out, row_stats=stats, kv=(1, 1))
    torch.cuda.synchronize()
    # group 1 alone: its columns are the full call's, group 0's columns and stats untouched
    assert torch.equal(out[:, 3072:], full[:, 3072:])
    assert torch.all(out[:, :3072].view(torch.int16) == SENTINEL)
    assert torch.equal(stats[12:], full_stats[12:]) and torch.all(stats[:12] == -7.0)
    B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                      causal=causal, out=out, row_stats=stats, kv=(0, 1))
    assert torch.equal(out, full) and torch.equal(stats, full_stats)


def test_prefill_split_plan_equals_full_call():
    """Four ranks of the plan (two KV groups x two causal row windows) reproduce the full
    causal pass at S = 2048, each window a call at its own q_base."""
    S = 2048
    inp = Inputs(SEED + 61, S, S)
    d = inp.dev()
    full = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S)
    out = _filled((S, 6144))
    for sh in shard.plan(4, S):
        r0, n = sh["row0"], sh["rows"]
        if n == 0:
            continue
        B.ga_attn_prefill(d["qg"][r0:r0 + n], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                          r0, r0 + n, out=out[r0:r0 + n],
                          kv=(sh["kv_first"], sh["kv_count"]))
    torch.cuda.synchronize()
    assert torch.equal(out, full)


def test_masked_groups_equal_full_call():
    S = 384
    inp = Inputs(SEED + 62, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 62, S, window=16, n_random=48)
    mask[9] = 0
    mcu = mask.cuda()
    f_out, f_w, f_h = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                       d["sin"], mcu, want_weights=True)
    out = _filled((S, 6144))
    w = _filled((24, S, S))
    hid = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mcu, out=out,
                     weights=w, hidden_rows=hid, kv=(0, 1))
    torch.cuda.synchronize()
    assert torch.equal(out[:, :3072], f_out[:, :3072]) and torch.equal(w[:12], f_w[:12])
    assert torch.all(out[:, 3072:].view(torch.int16) == SENTINEL)
    assert torch.all(w[12:].view(torch.int16) == SENTINEL)
    assert int(hid.item()) == int(f_h.item()) == 1
    B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mcu, out=out,
                     weights=w, hidden_rows=hid, kv=(1, 1))
    torch.cuda.synchronize()
    assert torch.equal(out, f_out) and torch.equal(w, f_w)
    assert int(hid.item()) == 1
