"""The entry points under CUDA-graph capture: after one ordinary call on the device (the
library's one-time set-up), a captured key prologue + prefill, a verify call and a
selection mask replay over new inputs written into the captured buffers, bit-identical to
direct calls on the same inputs."""
import pytest
import torch

from tests.parity import SEED
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


def _replay_matches(run, inputs, fresh_inputs):
    """Capture run() over `inputs` (static tensors), copy each fresh set in, replay, and
    compare with run() called directly on the fresh set."""
    run()                                   # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = run()
    for fresh in fresh_inputs:
        for dst, src in zip(inputs, fresh):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outs]
        want = run()
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)


def test_prefill_step_graph_replay():
    S = 384
    c, s = B.ga_rope_table_host(S)
    c, s = c.cuda(), s.cuda()
    sets = [synth.attention_inputs(SEED + 100 + i, S, S, device="cuda") for i in range(3)]
    qg, k, v, w_q, w_k = [t.clone() for t in sets[0]]
    k_prep = torch.empty_like(k)
    out = torch.empty(S, 24 * 256, dtype=torch.bfloat16, device="cuda")

    def run():
        B.ga_k_prologue(k, w_k, c, s, k_prep=k_prep)
        return [B.ga_attn_prefill(qg, k_prep, v, w_q, c, s, 0, S, out=out)]

    _replay_matches(run, [qg, k, v, w_q, w_k], sets[1:])


def test_verify_graph_replay():
    lens, rows, cap = [1000, 333], 16, 1040
    c, s = B.ga_rope_table_host(cap)
    c, s = c.cuda(), s.cuda()
    w_q = synth.normal_bf16(SEED + 110, "w_q", (256,), sigma=0.1, device="cuda")

    def make(i):
        kc = synth.normal_bf16(SEED + 111 + i, "k", (2, cap, 2, 256), device="cuda")
        vc = synth.normal_bf16(SEED + 111 + i, "v", (2, cap, 2, 256), device="cuda")
        qg = synth.normal_bf16(SEED + 111 + i, "qg", (2, rows, 24, 512), device="cuda")
        return qg, kc, vc

    sets = [make(i) for i in range(3)]
    qg, kc, vc = [t.clone() for t in sets[0]]
    out = torch.empty(2, rows, 24 * 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.ga_verify_workspace_bytes(2, rows, max(lens)), dtype=torch.uint8,
                     device="cuda")

    def run():
        return [B.ga_attn_verify(qg, kc, vc, lens, w_q, c, s, out=out, workspace=ws)]

    _replay_matches(run, [qg, kc, vc], sets[1:])


def test_select_graph_replay():
    T, k = 2048, 128
    sets = [(synth.block_scores(SEED + 120 + i, T, T // 4, device="cuda"),) for i in range(3)]
    scores = sets[0][0].clone()
    mask = torch.zeros(T, T, dtype=torch.uint8, device="cuda")

    def run():
        return [B.ga_select_mask(scores, T, k, mask=mask)]

    _replay_matches(run, [scores], sets[1:])
