"""GPU parity of the verify windows over e4m3 caches: bit-identical to the bf16 verify over
the widened rows bf16(fp32(code * scale)), and within tolerance of the oracle's quantize,
widen and attend."""
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


def _caches(seed, n, rows, cap):
    w_q = synth.normal_bf16(seed, "w_q", (256,), sigma=0.1, device="cuda")
    w_k = synth.normal_bf16(seed, "w_k", (256,), sigma=0.1, device="cuda")
    c, s = B.ga_rope_table_host(cap)
    c, s = c.cuda(), s.cuda()
    kd = torch.empty(n, cap, 2, 256, dtype=torch.bfloat16, device="cuda")
    vd = torch.stack([synth.normal_bf16(seed, "v", (cap, 2, 256), sub=b, device="cuda")
                      for b in range(n)])
    for b in range(n):
        k = synth.normal_bf16(seed, "k", (cap, 2, 256), sub=b, device="cuda")
        B.ga_k_prologue(k, w_k, c, s, k_prep=kd[b])
    qg = torch.stack([synth.normal_bf16(seed, "qg", (rows, 24, 512), sub=b, device="cuda")
                      for b in range(n)])
    return qg, kd, vd, w_q, (c, s)


def _widen(q, sc):
    """The GPU's codes and scales widened on the host with the oracle's formula."""
    return torch.from_numpy(O.dequantize_e4m3_rows(decode_e4m3(q.cpu().numpy()),
                                                   sc.cpu().numpy().astype(np.float64))
                            ).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("rows", [16, 1])
def test_e4m3_equals_bf16_verify_over_widened_rows(rows):
    """Ragged lengths from 0, windows ending inside a tile and at its end, 16-row verify and
    1-row decode: the e4m3 call's bits are the bf16 call's over the widened rows."""
    lens = [1000, 1537, 0, 383, 128 - rows]
    cap = 1600
    qg, kd, vd, w_q, (c, s) = _caches(SEED + 70 + rows, len(lens), rows, cap)
    kq, ksc = B.ga_kv_quantize_e4m3(kd)
    vq, vsc = B.ga_kv_quantize_e4m3(vd)
    got = B.ga_attn_verify_e4m3(qg, kq, ksc, vq, vsc, lens, w_q, c, s)
    want = B.ga_attn_verify(qg, _widen(kq, ksc), _widen(vq, vsc), lens, w_q, c, s)
    torch.cuda.synchronize()
    assert torch.equal(got, want), (got.float() - want.float()).abs().max()


def test_e4m3_against_oracle():
    """The oracle quantizes the prepared keys and the values, widens them and attends;
    sampled heads of two sequences, one of 9,000 cached keys split over several chunks."""
    lens, rows, cap = [9000, 700], 8, 9024
    qg, kd, vd, w_q, (c, s) = _caches(SEED + 72, len(lens), rows, cap)
    kq, ksc = B.ga_kv_quantize_e4m3(kd)
    vq, vsc = B.ga_kv_quantize_e4m3(vd)
    got = B.ga_attn_verify_e4m3(qg, kq, ksc, vq, vsc, lens, w_q, c, s)
    torch.cuda.synchronize()
    oc, os_ = O.rope_tables(cap)
    heads = [0, 11, 12, 23]
    for b, L in enumerate(lens):
        kc = O.dequantize_e4m3_rows(*O.quantize_e4m3_rows(np64(kd[b, :L + rows])))
        vc = O.dequantize_e4m3_rows(*O.quantize_e4m3_rows(np64(vd[b, :L + rows])))
        AttnRef(np64(qg[b]), kc, vc, np64(w_q), oc, os_, L, L + rows, "causal",
                heads=heads).check(got[b], what=f"e4m3 verify seq {b} L={L}")
