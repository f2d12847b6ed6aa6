"""The causal, bidirectional and stored-mask passes run as clusters of two CTAs that share
each key and value tile (two query heads of one KV group per pair item, cta_group::2 MMAs
issued by the even CTA). Every output, statistic and weight must be the same bits as the
single-CTA kernel's: the pair changes only which
SM's shared memory holds which half of a tile, not any arithmetic. The oracle checks of the
other GPU tests run through the default forms; these tests pin the two forms to each other
on ragged sizes, windows, KV groups and masks with hidden rows."""
import contextlib

import pytest
import torch

from tests.parity import SEED, Inputs
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


@contextlib.contextmanager
def _pairs(enable):
    prev = B.ga_debug_set_cta_pairs(enable)
    try:
        yield
    finally:
        B.ga_debug_set_cta_pairs(prev)


def _both(fn, mode=2):
    """fn() under single CTAs and under CTA pairs (mode 2: wherever the heads allow them,
    whatever the size); both results (tuples of tensors)."""
    with _pairs(0):
        single = fn()
        torch.cuda.synchronize()
    with _pairs(mode):
        paired = fn()
        torch.cuda.synchronize()
    assert B.ga_device_status() == 0
    return single, paired


def _equal(single, paired):
    for x, y in zip(single, paired):
        assert x.shape == y.shape
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)


def test_switch_round_trips():
    prev = B.ga_debug_set_cta_pairs(1)
    assert B.ga_debug_set_cta_pairs(2) == 1
    assert B.ga_debug_set_cta_pairs(0) == 2
    assert B.ga_debug_set_cta_pairs(prev) == 0


def test_default_mode_picks_by_keys():
    """Mode 1 (the default) runs a call over 1,024 keys on single CTAs and one over 2,048
    keys as pairs; at both sizes its output is the same bits as modes 0 and 2 give."""
    for S in (1024, 2048):
        inp = Inputs(SEED + 91, S, S)
        d = inp.dev()

        def run():
            return (B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                      d["sin"], 0, S),)

        with _pairs(1):
            default = run()
            torch.cuda.synchronize()
        single, paired = _both(run)
        _equal(single, default)
        _equal(paired, default)


@pytest.mark.parametrize("S,causal", [(64, True), (333, True), (333, False), (2048, True),
                                      (2048, False)])
def test_prefill_pairs_equal_single(S, causal):
    inp = Inputs(SEED + 90 + S % 7, S, S)
    d = inp.dev()

    def run():
        stats = torch.zeros(24, S, 2, device="cuda")
        out = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0,
                                S, causal=causal, row_stats=stats)
        return out, stats

    _equal(*_both(run))


@pytest.mark.parametrize("q_base,rows", [(128, 200), (960, 37), (64, 1)])
def test_window_pairs_equal_single(q_base, rows):
    T = q_base + rows
    inp = Inputs(SEED + 97, T, T)
    d = inp.dev()

    def run():
        out = B.ga_attn_prefill(d["qg"][q_base:], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                d["sin"], q_base, T)
        return (out,)

    _equal(*_both(run))


@pytest.mark.parametrize("kv", [(0, 1), (1, 1)])
def test_kv_group_pairs_equal_single(kv):
    S = 700
    inp = Inputs(SEED + 98, S, S)
    d = inp.dev()

    def run():
        out = torch.zeros(S, 6144, dtype=torch.bfloat16, device="cuda")
        B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, S,
                          out=out, kv=kv)
        return (out,)

    _equal(*_both(run))


@pytest.mark.parametrize("S,window,n_random", [(384, 16, 48), (1104, 128, 300)])
def test_masked_pairs_equal_single(S, window, n_random):
    inp = Inputs(SEED + 99, S, S)
    d = inp.dev()
    mask = synth.selection_mask(SEED + 99, S, window=window, n_random=n_random)
    mask[5] = 0          # a row with no visible key
    mask[128:256] = 0    # a whole row tile hidden: its items have no key tiles
    mcu = mask.cuda()

    def run():
        out, w, hidden = B.ga_attn_masked(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"],
                                          d["sin"], mcu, want_weights=True)
        return out, w, hidden

    _equal(*_both(run))
