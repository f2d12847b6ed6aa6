"""The tensor cores' fp32 accumulation error on the scores, measured: the band the parity
check allows for an ambiguous score rounding (tests/parity.py, TC_BAND_ULP32) must cover it
with room to spare.

The score is "the bf16 GEMM result" (pegainfer PR #1151, the commit that adds the attention
reader): the fp32 reduction order inside the tensor core is the hardware's own. This test
forms 2^20 dot products of (1+w)-normed bf16 rows (w = 0) through ga_debug_qk_fp32, which
issues the attention kernel's own S = Q K^T (tcgen05.mma, sixteen K16 steps), and compares
each with the exact dot product, in units of one fp32 ulp of the largest partial sum over
16-product groups (the unit the band is stated in)."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import SEED, TC_BAND_ULP32, _ulp32
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod
from verify_gated_gqa_gb300 import synth

pytestmark = pytest.mark.gpu

N_TILES = 64   # 64 x 128 x 128 = 2^20 dot products


def test_tensor_core_accumulation_error_inside_the_parity_band():
    build_mod.build()
    rows = N_TILES * 128
    q = O.rms_norm_1pw(synth.normal_bf16(SEED + 90, "qg", (rows, 256)).double().numpy(),
                       np.zeros(256))
    k = O.rms_norm_1pw(synth.normal_bf16(SEED + 90, "k", (rows, 256)).double().numpy(),
                       np.zeros(256))
    qd = torch.from_numpy(q).to(torch.bfloat16).view(N_TILES, 128, 256).cuda()
    kd = torch.from_numpy(k).to(torch.bfloat16).view(N_TILES, 128, 256).cuda()
    s = B.ga_debug_qk_fp32(qd, kd).double().cpu().numpy()
    assert B.ga_device_status() == 0
    q3, k3 = q.reshape(N_TILES, 128, 256), k.reshape(N_TILES, 128, 256)
    worst = 0.0
    for t in range(N_TILES):
        prods = q3[t][:, None, :] * k3[t][None, :, :]          # exact (bf16 x bf16)
        groups = prods.reshape(128, 128, 16, 16).sum(axis=3)   # exact in float64
        pref = np.cumsum(groups, axis=2)
        unit = _ulp32(np.max(np.abs(pref), axis=2))
        err = np.abs(s[t] - pref[:, :, -1]) / unit
        worst = max(worst, float(err.max()))
    print(f"[tc-error] 2^20 dot products: max error {worst:.3f} fp32 ulps of the largest "
          f"16-product partial sum (parity band {TC_BAND_ULP32})")
    assert worst <= TC_BAND_ULP32 / 1.5
