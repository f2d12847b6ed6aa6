"""The seeded generator: counter-based bits, slices and the selection-mask recipe."""
import numpy as np
import torch

from verify_gated_gqa_gb300 import synth


def _splitmix_ref(key, i):
    m = (1 << 64) - 1
    z = (key + (i + 1) * 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_counter_bits_match_integer_reference():
    key = synth.stream_key(20261101, "qg")
    idx = [0, 1, 2, 12345, 2 ** 31 + 7, 2 ** 40 + 3]
    for i in idx:
        got = int(synth.random_bits(key, i, 1)[0]) & ((1 << 64) - 1)
        assert got == _splitmix_ref(key, i)


def test_rows_slice_matches_whole_tensor():
    qg, *_ = synth.attention_inputs(7, 40, 40)
    assert torch.equal(synth.qg_rows(7, 13, 9), qg[13:22])


def test_normal_statistics():
    x = synth.normal_bf16(3, "v", (1 << 20,)).double()
    assert abs(x.mean().item()) < 5e-3 and abs(x.std().item() - 1) < 5e-3
    w = synth.normal_bf16(3, "w_q", (1 << 16,), sigma=0.1).double()
    assert abs(w.std().item() - 0.1) < 2e-3


def test_selection_mask_recipe():
    S, W, R = 1500, 128, 1024
    m = synth.selection_mask(5, S, W, R).numpy()
    assert np.all(np.triu(m, 1) == 0)                       # causal
    for i in [0, 1, 127, 128, 500, 1151, 1152, 1499]:
        row = np.nonzero(m[i])[0]
        assert len(row) == min(i + 1, W + R)
        assert np.all(m[i, max(0, i - W + 1):i + 1] == 1)   # the local window
    again = synth.selection_mask(5, S, W, R).numpy()
    assert np.array_equal(m, again)
