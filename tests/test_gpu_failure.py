"""Failure detection without a GPU fault: every wait in the library's kernels is bounded;
one that runs out records a status the host reads, and the context stays usable. The test
makes a wait run out on purpose (a barrier nothing arrives on) through the library's own
bounded wait."""
import pytest
import torch

from tests.parity import SEED, Inputs
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_reports_and_the_context_survives():
    build_mod.build()
    L = B.lib()
    assert torch.cuda.is_available()
    B.ga_device_status(clear=True)                       # start from a clean word
    assert L.ga_debug_wait_timeout(200_000, None) == 0   # about 0.1 ms at the SM clock
    assert B.ga_device_status(clear=True) == 1           # the wait gave up and said so
    assert B.ga_device_status(clear=True) == 0           # and the word was cleared
    # the context still works: a small causal pass matches the oracle
    inp = Inputs(SEED + 50, 64, 64)
    d = inp.dev()
    got = B.ga_attn_prefill(d["qg"], d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], 0, 64)
    inp.ref(0, 64, "causal").check(got, what="S=64 after a recorded wait timeout")
    assert B.ga_device_status() == 0
