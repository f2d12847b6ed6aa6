"""GPU parity of prefill over e4m3 caches: the widening kernel bit for bit against the
oracle's widening, the prefill call bit-identical to the bf16 prefill over the same widened
rows (causal, a prefix window, bidirectional), and within tolerance of the oracle's
quantize-widen-attend."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, AttnRef, np64
from tests.test_gpu_quant import decode_e4m3
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


def _host_widen(q, sc):
    """The device codes and scales widened on the host with the oracle's formula."""
    return torch.from_numpy(O.dequantize_e4m3_rows(decode_e4m3(q.cpu().numpy()),
                                                   sc.cpu().numpy().astype(np.float64))
                            ).to(torch.bfloat16)


def test_dequantize_matches_oracle():
    """Rows of very different magnitudes, a zero row and a row at the saturation point:
    every widened value equal to the oracle's bf16(fp32(code * scale))."""
    rng = np.random.default_rng(61)
    n = 700
    x = rng.normal(size=(n, 2, 256)) * 2.0 ** rng.integers(-20, 20, (n, 2, 1))
    x[3, 1] = 0.0
    x[5, 0, :4] = [448.0, -448.0, 1e-3, 3.0]
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    q, sc = B.ga_kv_quantize_e4m3(xt)
    got = B.ga_kv_dequantize_e4m3(q, sc)
    torch.cuda.synchronize()
    want = _host_widen(q, sc)
    assert torch.equal(got.cpu().view(torch.int16), want.view(torch.int16))
    assert bool((got[3, 1] == 0).all())


def _case(seed, S):
    qg, k, v, w_q, w_k = synth.attention_inputs(seed, S, S, device="cuda")
    c, s = B.ga_rope_table_host(S)
    c, s = c.cuda(), s.cuda()
    kd = B.ga_k_prologue(k, w_k, c, s)
    kq, ksc = B.ga_kv_quantize_e4m3(kd)
    vq, vsc = B.ga_kv_quantize_e4m3(v)
    return qg, w_q, (c, s), (kq, ksc, vq, vsc), (k, v, w_k)


@pytest.mark.parametrize("S,q_base,causal", [(2048, 0, True), (2048, 1024, True),
                                             (1536, 0, False), (700, 576, True)])
def test_prefill_e4m3_equals_bf16_prefill_over_widened_rows(S, q_base, causal):
    """A full causal pass, a prefix window, a bidirectional pass and a ragged T: the e4m3
    call's bits equal ga_attn_prefill's over the rows widened on the host."""
    qg, w_q, (c, s), (kq, ksc, vq, vsc), _ = _case(SEED + 80 + S + q_base, S)
    kw, vw = _host_widen(kq, ksc).cuda(), _host_widen(vq, vsc).cuda()
    rows = S - q_base
    win = qg[q_base:].contiguous()
    got = B.ga_attn_prefill_e4m3(win, kq, ksc, vq, vsc, w_q, c, s, q_base=q_base, T=S,
                                 causal=causal)
    want = B.ga_attn_prefill(win, kw, vw, w_q, c, s, q_base, S, causal=causal)
    torch.cuda.synchronize()
    assert got.shape == (rows, 24 * 256)
    assert torch.equal(got, want), (got.float() - want.float()).abs().max()


def test_prefill_e4m3_against_oracle():
    """The oracle quantizes the prepared keys and the values, widens them and attends;
    sampled heads of a causal S = 1024 pass."""
    S = 1024
    qg, w_q, (c, s), (kq, ksc, vq, vsc), (k, v, w_k) = _case(SEED + 86, S)
    got = B.ga_attn_prefill_e4m3(qg, kq, ksc, vq, vsc, w_q, c, s)
    torch.cuda.synchronize()
    oc, os_ = O.rope_tables(S)
    kp = O.prep_keys(np64(k), np64(w_k), oc, os_)
    kc = O.dequantize_e4m3_rows(*O.quantize_e4m3_rows(kp))
    vc = O.dequantize_e4m3_rows(*O.quantize_e4m3_rows(np64(v)))
    AttnRef(np64(qg), kc, vc, np64(w_q), oc, os_, 0, S, "causal",
            heads=[0, 11, 12, 23]).check(got, what="e4m3 prefill S=1024")


def test_prefill_e4m3_s8192_full_output():
    """The benchmark's size, causal S = 8192: every output of the e4m3 call equals the bf16
    prefill's over the rows widened on the host."""
    S = 8192
    qg, w_q, (c, s), (kq, ksc, vq, vsc), _ = _case(SEED + 87, S)
    kw, vw = _host_widen(kq, ksc).cuda(), _host_widen(vq, vsc).cuda()
    got = B.ga_attn_prefill_e4m3(qg, kq, ksc, vq, vsc, w_q, c, s)
    want = B.ga_attn_prefill(qg, kw, vw, w_q, c, s, 0, S)
    torch.cuda.synchronize()
    assert torch.equal(got, want), int((got != want).sum())
