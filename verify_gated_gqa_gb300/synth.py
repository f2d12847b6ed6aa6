"""Seeded synthetic inputs for gated GQA attention.

This module only draws numbers; it holds none of the attention arithmetic. Both the
CPU oracle (through the tests) and the CUDA path take their inputs from here, so the
two sides see identical bits.

Generator: every element is drawn independently from a counter-based stream.
SplitMix64's finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) maps (seed, tensor id, element index) to 64 random bits;
Box-Muller (1958) turns the two 32-bit halves into one N(0, 1) double, which is
scaled by sigma and rounded once (round-to-nearest-even) to bfloat16.

Workload shapes follow the pages' prefill and verify configurations: fused q|gate rows
[rows, 24, 512] (per head the first 256 values are q and the last 256 the gate), keys
and values [T, 2, 256], (1+w) norm weights [256] with w ~ N(0, 0.1).
"""
from __future__ import annotations

import torch

N_Q_HEADS = 24
N_KV_HEADS = 2
HEAD_DIM = 256

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# Tensor ids: part of the counter, so that tensors drawn with one seed are independent.
TENSOR_IDS = {"qg": 1, "k": 2, "v": 3, "w_q": 4, "w_k": 5, "mask": 6, "block_scores": 7}


def _to_i64(u: int) -> int:
    """Reinterpret an unsigned 64-bit constant as torch's signed int64."""
    u &= _MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns (torch's >> is arithmetic)."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 finaliser on int64 bit patterns (wrapping arithmetic)."""
    z = (z ^ _srl(z, 30)) * _to_i64(_M1)
    z = (z ^ _srl(z, 27)) * _to_i64(_M2)
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor: str, sub: int = 0) -> int:
    """64-bit key of one tensor's stream (sub distinguishes e.g. sequences)."""
    t = TENSOR_IDS[tensor]
    return _mix_int(_mix_int(seed + _GOLDEN) ^ (t * 0x100000001B3 + sub * 0xD1B54A32D192ED03))


def random_bits(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """64 random bits (as int64) for element indices start .. start+count-1."""
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    z = idx * _to_i64(_GOLDEN) + _to_i64(key + _GOLDEN)
    return _mix(z)


def _bits_to_normal(bits: torch.Tensor) -> torch.Tensor:
    hi = _srl(bits, 32).to(torch.float64)
    lo = (bits & 0xFFFFFFFF).to(torch.float64)
    u1 = (hi + 0.5) * (1.0 / 4294967296.0)
    u2 = (lo + 0.5) * (1.0 / 4294967296.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * torch.pi) * u2)


def _double_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round float64 to bfloat16 once (nearest, ties to even), no float32 detour."""
    m, e = torch.frexp(x)
    e = torch.clamp(e, min=-125)
    q = torch.ldexp(torch.round(torch.ldexp(x, (8 - e).to(torch.float64))), (e - 8).to(torch.float64))
    return q.to(torch.bfloat16)  # exact: q already holds a bfloat16 value


def normal_bf16(seed: int, tensor: str, shape, sigma: float = 1.0, sub: int = 0,
                device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """A bf16 tensor of the given shape with N(0, sigma^2) entries from the counter stream."""
    n = 1
    for s in shape:
        n *= int(s)
    key = stream_key(seed, tensor, sub)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        z = _bits_to_normal(random_bits(key, s, c, device))
        out[s:s + c] = _double_to_bf16(z * sigma)
    return out.view(*shape)


def block_scores(seed: int, rows: int, n_blocks: int, device="cpu", chunk: int = 1 << 24):
    """float32 [rows, n_blocks] N(0, 1) indexer block scores from the counter stream (each
    double rounded once to float32), standing in for the indexer's output."""
    n = rows * n_blocks
    key = stream_key(seed, "block_scores")
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        out[s:s + c] = _bits_to_normal(random_bits(key, s, c, device)).to(torch.float32)
    return out.view(rows, n_blocks)


def attention_inputs(seed: int, rows: int, T: int, device="cpu"):
    """qg [rows,24,512], k_raw [T,2,256], v [T,2,256], w_q [256], w_k [256] (all bf16).

    qg rows are the query window's rows (positions q_base .. q_base+rows-1 for the
    caller's q_base); k and v hold all T keys.
    """
    qg = normal_bf16(seed, "qg", (rows, N_Q_HEADS, 2 * HEAD_DIM), device=device)
    k = normal_bf16(seed, "k", (T, N_KV_HEADS, HEAD_DIM), device=device)
    v = normal_bf16(seed, "v", (T, N_KV_HEADS, HEAD_DIM), device=device)
    w_q = normal_bf16(seed, "w_q", (HEAD_DIM,), sigma=0.1, device=device)
    w_k = normal_bf16(seed, "w_k", (HEAD_DIM,), sigma=0.1, device=device)
    return qg, k, v, w_q, w_k


def qg_rows(seed: int, row0: int, nrows: int, device="cpu") -> torch.Tensor:
    """Rows row0 .. row0+nrows-1 of the qg tensor that attention_inputs draws (any size)."""
    per_row = N_Q_HEADS * 2 * HEAD_DIM
    key = stream_key(seed, "qg")
    z = _bits_to_normal(random_bits(key, row0 * per_row, nrows * per_row, device))
    return _double_to_bf16(z).view(nrows, N_Q_HEADS, 2 * HEAD_DIM)


def selection_mask(seed: int, S: int, window: int = 128, n_random: int = 1024,
                   device="cpu", block: int = 256) -> torch.Tensor:
    """uint8 [S, S] sparse-selection mask (non-zero = visible).

    Row i sees its causal local window max(0, i-window+1) .. i, plus n_random distinct
    keys drawn uniformly without replacement from 0 .. i-window (all of them when there
    are no more than n_random). The draw ranks each candidate key by 64 counter bits
    (seed, "mask", row i, key j) and keeps the n_random smallest.
    """
    mask = torch.zeros(S, S, dtype=torch.uint8, device=device)
    idx = torch.arange(S, device=device)
    local = (idx[None, :] <= idx[:, None]) & (idx[None, :] > idx[:, None] - window)
    mask[local] = 1
    key = stream_key(seed, "mask")
    for r0 in range(0, S, block):
        r1 = min(S, r0 + block)
        n_cand_max = max(0, r1 - 1 - window + 1)
        if n_cand_max == 0:
            continue
        rows = torch.arange(r0, r1, device=device)
        cols = torch.arange(n_cand_max, device=device)
        lin = rows[:, None] * S + cols[None, :]
        bits = _mix(lin * _to_i64(_GOLDEN) + _to_i64(key + _GOLDEN))
        n_cand = (rows - window + 1).clamp(min=0)
        valid = cols[None, :] < n_cand[:, None]
        big = torch.iinfo(torch.int64).max
        rank = torch.where(valid, bits, torch.full_like(bits, big))
        kk = min(n_random, n_cand_max)
        sel = torch.topk(rank, kk, dim=1, largest=False, sorted=False).indices
        take = torch.gather(valid, 1, sel)
        rr = rows[:, None].expand_as(sel)
        mask[rr[take], sel[take]] = 1
    return mask
