"""The parity check itself (CPU): an alternative rounding of an ambiguous score is
accepted; a genuine error of the same size elsewhere is not."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import AttnRef, Inputs, _alternatives


def _case():
    inp = Inputs(4242, 96, 96, device="cpu")
    ref = inp.ref(0, 96, "causal", want_weights=True)
    return inp, ref


def _find_ambiguous(ref):
    for i in range(len(ref.rows)):
        for h in ref.heads:
            idx = np.nonzero(ref.vis[i])[0]
            dot, b, alt = _alternatives(ref.q_hat[i, h], ref.k_hat[idx, h // 12], None)
            for j in np.nonzero(~np.isnan(alt))[0]:
                return i, h, idx, j, alt[j]
    return None


def _row_with_score(ref, i, h, idx, j, new_score):
    kv = h // 12
    s = O.scores(ref.q_hat[i:i + 1, h], ref.k_hat[idx, kv])[0]
    s[j] = new_score / 16.0
    w_hat = O.bf16_sig(np.exp(s))
    L = w_hat.sum()
    o = O.bf16((w_hat @ ref.v[idx, kv]) / L)
    return O.bf16(o * O.sigmoid_gate(ref.gate[i, h]))


def test_alternative_rounding_is_accepted():
    inp, ref = _case()
    found = _find_ambiguous(ref)
    assert found is not None
    i, h, idx, j, alt = found
    got = ref.out.copy()
    got[i, h * 256:(h + 1) * 256] = _row_with_score(ref, i, h, idx, j, alt)
    ref.check(torch.from_numpy(got), None, "alternative rounding")


def test_genuine_error_is_rejected():
    inp, ref = _case()
    got = ref.out.copy()
    i, h = 40, 5
    idx = np.nonzero(ref.vis[i])[0]
    kv = h // 12
    s = O.scores(ref.q_hat[i:i + 1, h], ref.k_hat[idx, kv])[0]
    j = int(np.argmax(s))
    # a 1% error on the largest score of the row: not a rounding ambiguity
    row = _row_with_score(ref, i, h, idx, j, O.bf16(s[j] * 16.0 * 1.06))
    got[i, h * 256:(h + 1) * 256] = row
    assert not np.array_equal(row, ref.out[i, h * 256:(h + 1) * 256])
    with pytest.raises(AssertionError):
        ref.check(torch.from_numpy(got), None, "planted genuine error (must fail)")


def test_wrong_kv_head_is_rejected():
    inp, ref = _case()
    got = ref.out.copy()
    got[:, :256] = ref.out[:, 12 * 256:13 * 256]    # head 0 answered with head 12's output
    with pytest.raises(AssertionError):
        ref.check(torch.from_numpy(got), None, "planted swapped head (must fail)")
