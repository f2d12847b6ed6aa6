"""The allocation-free masked entry point (ga_attn_masked_static): its refusals, and on the
GPU its results against ga_attn_masked on the same inputs, two different calls in a row.

The entry point has no counterpart in the pages; its results must be those of the
workspace-taking call it stands in for."""
import ctypes

import numpy as np
import pytest
import torch

from tests.parity import SEED, Inputs
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import synth

A = 0x10000        # a 16-byte-aligned fake device address (never dereferenced)
MIS = 0x10002


def _static(L, rows=256, T=1024, q_base=0, mask=A, ld=1024, qg=A, out=A):
    return L.ga_attn_masked_static(qg, A, A, A, A, A, 100000, rows, T, q_base, mask, ld, out,
                                   None, None, None)


def test_static_refusals_make_no_cuda_call():
    L = B.lib()
    before = L.ga_debug_cuda_calls()
    assert _static(L, qg=None) == -1                       # NULL
    assert _static(L, q_base=32) == -4                     # RANGE
    assert _static(L, mask=MIS) == -3                      # ALIGN
    assert _static(L, T=9000, ld=9008) == -4               # beyond the masked cap
    assert _static(L, rows=0) == 0                         # nothing to do
    # beyond the static scratch: 8192 rows x 8192 keys needs ~110 MB of scratch
    assert B.ga_masked_workspace_bytes(8192, 8192) > 16 << 20
    assert _static(L, rows=8192, T=8192, ld=8192) == -6    # WORKSPACE, before any CUDA call
    assert L.ga_debug_cuda_calls() == before


def _case(seed, rows, T, q_base, window, n_random):
    inp = Inputs(seed, q_base + rows, T)
    d = inp.dev()
    mask = synth.selection_mask(seed, T, window=window, n_random=n_random)[q_base:q_base + rows]
    # pad the mask rows to a 16-byte multiple leading dimension
    ld = (T + 15) // 16 * 16
    m = torch.zeros(rows, ld, dtype=torch.uint8)
    m[:, :T] = mask
    return d, m.cuda(), q_base, T


@pytest.mark.gpu
def test_static_matches_workspace_call_two_calls_in_a_row():
    cases = [_case(SEED + 40, 256, 256, 0, 32, 64), _case(SEED + 41, 200, 333, 128, 16, 40)]
    for d, mask, q_base, T in cases:
        rows = mask.shape[0]
        qg = d["qg"][q_base:q_base + rows]
        ref_out, ref_w, ref_h = B.ga_attn_masked(qg, d["k_prep"], d["v"], d["w_q"], d["cos"],
                                                 d["sin"], mask, q_base=q_base, T=T,
                                                 want_weights=True)
        out = torch.empty_like(ref_out)
        w = torch.empty_like(ref_w)
        hid = torch.zeros(1, dtype=torch.int32, device=out.device)
        B.ga_attn_masked_static(qg, d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mask,
                                out, hid, weights=w, q_base=q_base, T=T)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: equal bit for bit (a tolerance of zero)
        assert torch.equal(out, ref_out)
        assert torch.equal(w, ref_w)
        assert int(hid.item()) == int(ref_h.item())
    assert B.ga_device_status() == 0


@pytest.mark.gpu
def test_static_at_the_size_limit():
    """The largest call the static scratch takes at T = 8192 (1,239 rows: the scratch's
    last rows in use) against the workspace call, bit for bit, so the layout's end stays
    inside the array; one row more is refused."""
    T, rows, q_base = 8192, 1239, 6912
    assert B.ga_masked_workspace_bytes(rows, T) <= 16 << 20 < B.ga_masked_workspace_bytes(rows + 1, T)
    d, mask, q_base, T = _case(SEED + 42, rows, T, q_base, 128, 1024)
    qg = d["qg"][q_base:q_base + rows]
    ref_out, _, ref_h = B.ga_attn_masked(qg, d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"],
                                         mask, q_base=q_base, T=T)
    out = torch.empty_like(ref_out)
    hid = torch.zeros(1, dtype=torch.int32, device=out.device)
    B.ga_attn_masked_static(qg, d["k_prep"], d["v"], d["w_q"], d["cos"], d["sin"], mask, out,
                            hid, q_base=q_base, T=T)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert int(hid.item()) == int(ref_h.item()) == 0
    big = torch.zeros(rows + 1, T, dtype=torch.uint8, device=out.device)
    with pytest.raises(B.GaError, match="WORKSPACE"):
        B.ga_attn_masked_static(d["qg"][q_base - 64:q_base + rows], d["k_prep"], d["v"], d["w_q"],
                                d["cos"], d["sin"], big,
                                torch.empty(rows + 1, 6144, dtype=torch.bfloat16,
                                            device=out.device), hid, q_base=q_base - 64, T=T)
    assert B.ga_device_status() == 0
