"""GPU parity of the e4m3 cache-row quantizer: every scale bit for bit and every code equal
to the oracle's, on rows of very different magnitudes, a zero row and rows at ties."""
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from tests.parity import np64
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import build as build_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.lib()
    yield
    assert B.ga_device_status() == 0


def decode_e4m3(codes):
    """Byte codes -> values, from the format's definition (sign, 4-bit exponent with bias 7,
    3-bit mantissa, subnormals when the exponent field is 0)."""
    c = np.asarray(codes, np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e, m = (c >> 3) & 15, c & 7
    val = np.where(e == 0, m / 8 * 2.0 ** -6, (1 + m / 8) * 2.0 ** (e - 7.0))
    assert not np.any((e == 15) & (m == 7)), "NaN code"
    return sign * val


def test_quantize_matches_oracle():
    rng = np.random.default_rng(60)
    n = 600
    x = rng.normal(size=(n, 2, 256)) * 2.0 ** rng.integers(-20, 20, (n, 2, 1))
    x[3, 1] = 0.0                                   # a zero row
    x[4, 0, :] = 1e-3                               # a constant row: every element at 448
    x[5, 0, :8] = [448.0, 1.0625, 1.1875, -3.0, 0.5, -448.0, 2.0 ** -9, 1000.0]
    xt = torch.from_numpy(x).to(torch.bfloat16)
    q, sc = B.ga_kv_quantize_e4m3(xt.cuda())
    torch.cuda.synchronize()
    want_q, want_sc = O.quantize_e4m3_rows(np64(xt))
    got_sc = sc.cpu().numpy().astype(np.float64)
    assert np.array_equal(got_sc, want_sc), np.flatnonzero(got_sc != want_sc)[:5]
    got_q = decode_e4m3(q.cpu().numpy())
    bad = np.flatnonzero(got_q.reshape(-1) != want_q.reshape(-1))
    assert bad.size == 0, (bad[:5], got_q.reshape(-1)[bad[:5]], want_q.reshape(-1)[bad[:5]])
    assert got_sc[3, 1] == 0 and np.all(got_q[3, 1] == 0)
    assert np.all(np.abs(got_q[4, 0]) == 448.0)
