"""ctypes binding of libga_attn.so (the C ABI in include/ga_attn.h).

Argument marshalling only: every step of the attention runs in the library's CUDA
kernels. Tensors are torch tensors on the current CUDA device; the work goes on torch's
current stream. There is no CPU fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libga_attn.so")

N_Q_HEADS, N_KV_HEADS, HEAD_DIM, ROPE_DIMS = 24, 2, 256, 64
MASKED_MAX_TOKENS = 8192

STATUS = {0: "GA_OK", -1: "GA_ERR_NULL", -2: "GA_ERR_SHAPE", -3: "GA_ERR_ALIGN",
          -4: "GA_ERR_RANGE", -5: "GA_ERR_TABLE", -6: "GA_ERR_WORKSPACE",
          -7: "GA_ERR_DEVICE", -8: "GA_ERR_CUDA", -9: "GA_ERR_GEOMETRY"}

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_SZ = ctypes.c_size_t

# name: (restype, argtypes)
_SIGS = {
    "ga_abi_version": (_I, []),
    "ga_check_geometry": (_I, [_P]),
    "ga_status_string": (ctypes.c_char_p, [_I]),
    "ga_last_cuda_error": (_I, []),
    "ga_debug_cuda_calls": (ctypes.c_ulonglong, []),
    "ga_device_status": (_I, [_P, _I]),
    "ga_rope_table_host": (_I, [_I, _P, _P]),
    "ga_k_prologue": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "ga_q_prologue": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "ga_qk_prologue": (_I, [_P, _P, _I, _I, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P]),
    "ga_debug_wait_timeout": (_I, [_LL, _P]),
    "ga_debug_qk_fp32": (_I, [_P, _P, _I, _P, _P]),
    "ga_debug_set_cta_pairs": (_I, [_I]),
    "ga_attn_prefill": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "ga_attn_prefill_prepared": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "ga_attn_prefill_kv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "ga_attn_masked_kv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _LL, _I, _I, _P, _P,
                               _P, _P, _SZ, _P]),
    "ga_attn_masked_static": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _LL, _P, _P, _P,
                                   _P]),
    "ga_masked_workspace_bytes": (_SZ, [_I, _I]),
    "ga_attn_masked_prepared": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _LL, _P, _P, _P, _P, _SZ,
                                     _P]),
    "ga_attn_masked": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _LL, _P, _P, _P, _P,
                            _SZ, _P]),
    "ga_verify_workspace_bytes": (_SZ, [_I, _I, _I]),
    "ga_attn_verify": (_I, [_P, _P, _P, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P, _SZ, _P]),
    "ga_attn_verify_paged": (_I, [_P, _P, _P, _I, _I, _P, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P,
                                  _SZ, _P]),
    "ga_attn_prefill_batch": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _P, _I, _P, _P, _P, _I, _P,
                                   _P]),
    "ga_kv_quantize_e4m3": (_I, [_P, _LL, _P, _P, _P]),
    "ga_attn_verify_e4m3": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P, _SZ,
                                 _P]),
    "ga_select_mask": (_I, [_P, _LL, _I, _I, _I, _I, _P, _LL, _P]),
    "ga_kv_dequantize_e4m3": (_I, [_P, _P, _LL, _P, _P]),
    "ga_prefill_e4m3_workspace_bytes": (_SZ, [_I]),
    "ga_attn_prefill_e4m3": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P,
                                  _SZ, _P]),
}


class GaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == -8 and _lib is not None:
            extra = f" (cudaError {_lib.ga_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS.get(status, status)}{extra}")


class Geometry(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("rope_dims", ctypes.c_int),
                ("eps", ctypes.c_float), ("rope_base", ctypes.c_double)]


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run verify_gated_gqa_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(st: int, where: str):
    if st != 0:
        raise GaError(st, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _bf16_cuda(name, t, shape=None):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


# ------------------------------------------------------------------ host helpers
def ga_abi_version() -> int:
    return lib().ga_abi_version()


def ga_check_geometry(n_q_heads=24, n_kv_heads=2, head_dim=256, rope_dims=64, eps=1e-6,
                      rope_base=1e7) -> int:
    g = Geometry(n_q_heads, n_kv_heads, head_dim, rope_dims, eps, rope_base)
    return lib().ga_check_geometry(ctypes.byref(g))


def ga_status_string(status: int) -> str:
    return lib().ga_status_string(status).decode()


def ga_debug_cuda_calls() -> int:
    return lib().ga_debug_cuda_calls()


def ga_debug_set_cta_pairs(mode) -> int:
    """0 (or False): every pass on single CTAs; 2: the causal, bidirectional, stored-mask
    and batched passes as CTA pairs; 1 (or True, the default): the same, but single CTAs for
    calls over fewer than 2,048 keys (batches excepted). The same bits either way. Returns
    the previous mode."""
    st = lib().ga_debug_set_cta_pairs(int(mode))
    if st < 0:
        _check(st, "ga_debug_set_cta_pairs")
    return st


def ga_device_status(clear: bool = True) -> int:
    v = ctypes.c_int(0)
    _check(lib().ga_device_status(ctypes.byref(v), 1 if clear else 0), "ga_device_status")
    return v.value


def ga_rope_table_host(n_pos: int):
    """(cos, sin) bf16 CPU tensors [n_pos, 32] built by the library's host helper."""
    c = torch.empty(n_pos, ROPE_DIMS // 2, dtype=torch.int16)
    s = torch.empty(n_pos, ROPE_DIMS // 2, dtype=torch.int16)
    _check(lib().ga_rope_table_host(n_pos, _ptr(c), _ptr(s)), "ga_rope_table_host")
    return c.view(torch.bfloat16), s.view(torch.bfloat16)


# ------------------------------------------------------------------ device entry points
def ga_k_prologue(k_raw, w_k, cos_tab, sin_tab, pos_base=0, k_prep=None):
    _bf16_cuda("k_raw", k_raw)
    n_tok = k_raw.shape[0]
    if k_prep is None:
        k_prep = torch.empty_like(k_raw)
    for n, t in (("w_k", w_k), ("cos_tab", cos_tab), ("sin_tab", sin_tab), ("k_prep", k_prep)):
        _bf16_cuda(n, t)
    _check(lib().ga_k_prologue(_ptr(k_raw), _ptr(w_k), _ptr(cos_tab), _ptr(sin_tab),
                               cos_tab.shape[0], n_tok, pos_base, _ptr(k_prep), _stream()),
           "ga_k_prologue")
    return k_prep


def ga_q_prologue(qg, w_q, cos_tab, sin_tab, q_base=0, q_prep=None):
    """Prepared queries [rows, 24, 256] (bf16(rope(norm(q)))) of the fused rows qg."""
    _bf16_cuda("qg", qg)
    rows = qg.shape[0]
    if q_prep is None:
        q_prep = torch.empty(rows, N_Q_HEADS, HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    for n, t in (("w_q", w_q), ("cos_tab", cos_tab), ("sin_tab", sin_tab), ("q_prep", q_prep)):
        _bf16_cuda(n, t)
    _check(lib().ga_q_prologue(_ptr(qg), _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab),
                               cos_tab.shape[0], rows, q_base, _ptr(q_prep), _stream()),
           "ga_q_prologue")
    return q_prep


def ga_qk_prologue(k_raw, w_k, qg, w_q, cos_tab, sin_tab, k_pos_base=0, q_base=0, k_prep=None,
                   q_prep=None):
    """Both prologues in one launch: (k_prep [n_tok, 2, 256], q_prep [rows, 24, 256]), the
    same bits as ga_k_prologue and ga_q_prologue."""
    _bf16_cuda("k_raw", k_raw)
    _bf16_cuda("qg", qg)
    n_tok, rows = k_raw.shape[0], qg.shape[0]
    if k_prep is None:
        k_prep = torch.empty_like(k_raw)
    if q_prep is None:
        q_prep = torch.empty(rows, N_Q_HEADS, HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    for n, t in (("w_k", w_k), ("w_q", w_q), ("cos_tab", cos_tab), ("sin_tab", sin_tab),
                 ("k_prep", k_prep), ("q_prep", q_prep)):
        _bf16_cuda(n, t)
    _check(lib().ga_qk_prologue(_ptr(k_raw), _ptr(w_k), n_tok, k_pos_base, _ptr(k_prep), _ptr(qg),
                                _ptr(w_q), rows, q_base, _ptr(q_prep), _ptr(cos_tab),
                                _ptr(sin_tab), cos_tab.shape[0], _stream()),
           "ga_qk_prologue")
    return k_prep, q_prep


def ga_attn_prefill_prepared(q_prep, qg, k_prep, v, q_base=0, T=None, causal=True, out=None,
                             row_stats=None):
    rows = qg.shape[0]
    T = k_prep.shape[0] if T is None else T
    if out is None:
        out = torch.empty(rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    for n, t in (("q_prep", q_prep), ("qg", qg), ("k_prep", k_prep), ("v", v), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_prefill_prepared(_ptr(q_prep), _ptr(qg), _ptr(k_prep), _ptr(v), rows, T,
                                          q_base, 1 if causal else 0, _ptr(out), _ptr(row_stats),
                                          _stream()),
           "ga_attn_prefill_prepared")
    return out


def ga_attn_prefill(qg, k_prep, v, w_q, cos_tab, sin_tab, q_base=0, T=None, causal=True,
                    out=None, row_stats=None, kv=None):
    """kv = (kv_first, kv_count) runs ga_attn_prefill_kv: only the query heads of those KV
    heads, whose output columns alone are written."""
    rows = qg.shape[0]
    T = k_prep.shape[0] if T is None else T
    if out is None:
        out = torch.empty(rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    for n, t in (("qg", qg), ("k_prep", k_prep), ("v", v), ("w_q", w_q), ("cos_tab", cos_tab),
                 ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    args = (_ptr(qg), _ptr(k_prep), _ptr(v), _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab),
            cos_tab.shape[0], rows, T, q_base, 1 if causal else 0)
    tail = (_ptr(out), _ptr(row_stats), _stream())
    if kv is None:
        _check(lib().ga_attn_prefill(*args, *tail), "ga_attn_prefill")
    else:
        _check(lib().ga_attn_prefill_kv(*args, int(kv[0]), int(kv[1]), *tail),
               "ga_attn_prefill_kv")
    return out


def ga_masked_workspace_bytes(rows: int, T: int) -> int:
    return lib().ga_masked_workspace_bytes(rows, T)


def ga_attn_masked(qg, k_prep, v, w_q, cos_tab, sin_tab, mask, q_base=0, T=None,
                   want_weights=False, out=None, weights=None, hidden_rows=None,
                   workspace=None, kv=None):
    """Returns (out, weights or None, hidden_rows int32 device tensor [1]). kv =
    (kv_first, kv_count) runs ga_attn_masked_kv (those KV heads' query heads only)."""
    rows = qg.shape[0]
    T = k_prep.shape[0] if T is None else T
    dev = qg.device
    if out is None:
        out = torch.empty(rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=dev)
    if want_weights and weights is None:
        weights = torch.empty(N_Q_HEADS, rows, T, dtype=torch.bfloat16, device=dev)
    if hidden_rows is None:
        hidden_rows = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = ga_masked_workspace_bytes(rows, T)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    if mask.dtype != torch.uint8 or not mask.is_cuda or mask.stride(1) != 1:
        raise ValueError("mask must be a uint8 CUDA tensor with unit column stride")
    for n, t in (("qg", qg), ("k_prep", k_prep), ("v", v), ("w_q", w_q), ("cos_tab", cos_tab),
                 ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    head = (_ptr(qg), _ptr(k_prep), _ptr(v), _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab),
            cos_tab.shape[0], rows, T, q_base, _ptr(mask), mask.stride(0))
    tail = (_ptr(out), _ptr(weights), _ptr(hidden_rows), _ptr(workspace), workspace.numel(),
            _stream())
    if kv is None:
        _check(lib().ga_attn_masked(*head, *tail), "ga_attn_masked")
    else:
        _check(lib().ga_attn_masked_kv(*head, int(kv[0]), int(kv[1]), *tail), "ga_attn_masked_kv")
    return out, weights, hidden_rows


def ga_attn_masked_prepared(q_prep, qg, k_prep, v, mask, q_base=0, T=None, want_weights=False,
                            out=None, weights=None, hidden_rows=None, workspace=None):
    """ga_attn_masked from prepared queries q_prep [rows, 24, 256] (ga_q_prologue's output):
    the mask prepass and the attention only. Returns (out, weights or None, hidden_rows)."""
    rows = qg.shape[0]
    T = k_prep.shape[0] if T is None else T
    dev = qg.device
    if out is None:
        out = torch.empty(rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=dev)
    if want_weights and weights is None:
        weights = torch.empty(N_Q_HEADS, rows, T, dtype=torch.bfloat16, device=dev)
    if hidden_rows is None:
        hidden_rows = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(ga_masked_workspace_bytes(rows, T), 1), dtype=torch.uint8,
                                device=dev)
    if mask.dtype != torch.uint8 or not mask.is_cuda or mask.stride(1) != 1:
        raise ValueError("mask must be a uint8 CUDA tensor with unit column stride")
    for n, t in (("q_prep", q_prep), ("qg", qg), ("k_prep", k_prep), ("v", v), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_masked_prepared(_ptr(q_prep), _ptr(qg), _ptr(k_prep), _ptr(v), rows, T,
                                         q_base, _ptr(mask), mask.stride(0), _ptr(out),
                                         _ptr(weights), _ptr(hidden_rows), _ptr(workspace),
                                         workspace.numel(), _stream()),
           "ga_attn_masked_prepared")
    return out, weights, hidden_rows


def ga_debug_qk_fp32(q, k):
    """Test hook: the tensor cores' fp32 dot products s[n, i, j] = q[n, i] . k[n, j] of bf16
    tiles q, k [n, 128, 256], formed as the attention kernel forms its scores."""
    for n, t in (("q", q), ("k", k)):
        _bf16_cuda(n, t)
    if q.dim() != 3 or tuple(q.shape[1:]) != (128, HEAD_DIM) or q.shape != k.shape:
        raise ValueError("q and k must both be [n, 128, 256]")
    s = torch.empty(q.shape[0], 128, 128, dtype=torch.float32, device=q.device)
    _check(lib().ga_debug_qk_fp32(_ptr(q), _ptr(k), q.shape[0], _ptr(s), _stream()),
           "ga_debug_qk_fp32")
    return s


def ga_select_mask(block_scores, T, block_topk, q_base=0, mask=None):
    """block_scores float32 [rows, >= ceil(T / 4)] (unit column stride) -> the selection
    mask uint8 [rows, ld] that ga_attn_masked reads (ld = T rounded up to 16 when the mask is
    allocated here; its columns from T on stay 0)."""
    if (block_scores.dtype != torch.float32 or not block_scores.is_cuda or
            block_scores.dim() != 2 or block_scores.stride(1) != 1):
        raise ValueError("block_scores must be a 2-D float32 CUDA tensor with unit column stride")
    rows = block_scores.shape[0]
    if mask is None:
        mask = torch.zeros(rows, (T + 15) // 16 * 16, dtype=torch.uint8,
                           device=block_scores.device)
    if (mask.dtype != torch.uint8 or not mask.is_cuda or mask.dim() != 2 or
            mask.shape[0] != rows or mask.stride(1) != 1):
        raise ValueError("mask must be a uint8 CUDA tensor [rows, ld] with unit column stride")
    _check(lib().ga_select_mask(_ptr(block_scores), block_scores.stride(0), rows, T, q_base,
                                block_topk, _ptr(mask), mask.stride(0), _stream()),
           "ga_select_mask")
    return mask


def ga_attn_masked_static(qg, k_prep, v, w_q, cos_tab, sin_tab, mask, out, hidden_rows,
                          weights=None, q_base=0, T=None):
    """The allocation-free masked call: the caller passes every output buffer (out,
    hidden_rows and, when weights are wanted, weights); the library uses its static scratch."""
    rows = qg.shape[0]
    T = k_prep.shape[0] if T is None else T
    if mask.dtype != torch.uint8 or not mask.is_cuda or mask.stride(1) != 1:
        raise ValueError("mask must be a uint8 CUDA tensor with unit column stride")
    for n, t in (("qg", qg), ("k_prep", k_prep), ("v", v), ("w_q", w_q), ("cos_tab", cos_tab),
                 ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_masked_static(_ptr(qg), _ptr(k_prep), _ptr(v), _ptr(w_q), _ptr(cos_tab),
                                       _ptr(sin_tab), cos_tab.shape[0], rows, T, q_base,
                                       _ptr(mask), mask.stride(0), _ptr(out), _ptr(weights),
                                       _ptr(hidden_rows), _stream()),
           "ga_attn_masked_static")
    return out, weights, hidden_rows


def ga_verify_workspace_bytes(n_seq: int, rows: int, max_len: int) -> int:
    return lib().ga_verify_workspace_bytes(n_seq, rows, max_len)


def ga_attn_verify(qg, k_cache, v_cache, seq_len, w_q, cos_tab, sin_tab, out=None,
                   workspace=None):
    """qg [n_seq, rows, 24, 512]; k_cache, v_cache [n_seq, cap, 2, 256]; seq_len: ints."""
    n_seq, rows = qg.shape[0], qg.shape[1]
    cap = k_cache.shape[1]
    lens = (ctypes.c_int * n_seq)(*[int(x) for x in seq_len])
    dev = qg.device
    if out is None:
        out = torch.empty(n_seq, rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws_bytes = ga_verify_workspace_bytes(n_seq, rows, max(int(x) for x in seq_len))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    for n, t in (("qg", qg), ("k_cache", k_cache), ("v_cache", v_cache), ("w_q", w_q),
                 ("cos_tab", cos_tab), ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_verify(_ptr(qg), _ptr(k_cache), _ptr(v_cache), cap, lens, n_seq, rows,
                                _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab), cos_tab.shape[0],
                                _ptr(out), _ptr(workspace), workspace.numel(), _stream()),
           "ga_attn_verify")
    return out


def ga_attn_verify_paged(qg, k_pages, v_pages, page_table, seq_len, w_q, cos_tab, sin_tab,
                         out=None, workspace=None):
    """qg [n_seq, rows, 24, 512]; k_pages, v_pages [n_pages, page_size, 2, 256];
    page_table int32 [n_seq, max_pages] on the device; seq_len: ints (host)."""
    n_seq, rows = qg.shape[0], qg.shape[1]
    n_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    if (page_table.dtype != torch.int32 or not page_table.is_cuda or page_table.dim() != 2
            or not page_table.is_contiguous() or page_table.shape[0] != n_seq):
        raise ValueError("page_table must be a contiguous int32 CUDA tensor [n_seq, max_pages]")
    if tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages and v_pages must have the same shape")
    lens = (ctypes.c_int * n_seq)(*[int(x) for x in seq_len])
    dev = qg.device
    if out is None:
        out = torch.empty(n_seq, rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws_bytes = ga_verify_workspace_bytes(n_seq, rows, max(int(x) for x in seq_len))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    for n, t in (("qg", qg), ("k_pages", k_pages), ("v_pages", v_pages), ("w_q", w_q),
                 ("cos_tab", cos_tab), ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_verify_paged(_ptr(qg), _ptr(k_pages), _ptr(v_pages), n_pages, page_size,
                                      _ptr(page_table), page_table.shape[1], lens, n_seq, rows,
                                      _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab), cos_tab.shape[0],
                                      _ptr(out), _ptr(workspace), workspace.numel(), _stream()),
           "ga_attn_verify_paged")
    return out


def ga_attn_prefill_batch(qg, row_start, q_base, k_pages, v_pages, page_table, w_q, cos_tab,
                          sin_tab, out=None):
    """qg [total_rows, 24, 512] packed; row_start: n_seq + 1 ints; q_base: n_seq ints (host);
    k_pages, v_pages [n_pages, page_size, 2, 256]; page_table int32 [n_seq, max_pages] on the
    device. Returns out [total_rows, 24*256]."""
    n_seq = len(q_base)
    if len(row_start) != n_seq + 1:
        raise ValueError("row_start needs n_seq + 1 entries")
    n_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    if (page_table.dtype != torch.int32 or not page_table.is_cuda or page_table.dim() != 2
            or not page_table.is_contiguous() or page_table.shape[0] != n_seq):
        raise ValueError("page_table must be a contiguous int32 CUDA tensor [n_seq, max_pages]")
    if tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages and v_pages must have the same shape")
    starts = (ctypes.c_int * (n_seq + 1))(*[int(x) for x in row_start])
    bases = (ctypes.c_int * max(n_seq, 1))(*[int(x) for x in q_base])
    total = qg.shape[0]
    if out is None:
        out = torch.empty(total, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    for n, t in (("qg", qg), ("k_pages", k_pages), ("v_pages", v_pages), ("w_q", w_q),
                 ("cos_tab", cos_tab), ("sin_tab", sin_tab), ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_prefill_batch(_ptr(qg), starts, bases, n_seq, _ptr(k_pages),
                                       _ptr(v_pages), n_pages, page_size, _ptr(page_table),
                                       page_table.shape[1], _ptr(w_q), _ptr(cos_tab),
                                       _ptr(sin_tab), cos_tab.shape[0], _ptr(out), _stream()),
           "ga_attn_prefill_batch")
    return out


def ga_kv_quantize_e4m3(x, q=None, scale=None):
    """x [..., 2, 256] bf16 (rows of prepared keys or values) -> (q uint8 [..., 2, 256],
    scale fp32 [..., 2])."""
    _bf16_cuda("x", x)
    if x.shape[-2:] != (N_KV_HEADS, HEAD_DIM):
        raise ValueError("x must end in [2, 256]")
    n_tok = x.numel() // (N_KV_HEADS * HEAD_DIM)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if q.dtype != torch.uint8 or not q.is_contiguous() or q.shape != x.shape:
        raise ValueError("q must be a contiguous uint8 tensor shaped like x")
    if scale.dtype != torch.float32 or not scale.is_contiguous() or scale.shape != x.shape[:-1]:
        raise ValueError("scale must be a contiguous float32 tensor shaped like x[..., 0]")
    _check(lib().ga_kv_quantize_e4m3(_ptr(x), n_tok, _ptr(q), _ptr(scale), _stream()),
           "ga_kv_quantize_e4m3")
    return q, scale


def ga_kv_dequantize_e4m3(q, scale, out=None):
    """q uint8 [..., 2, 256] e4m3 codes, scale fp32 [..., 2] -> the widened rows, bf16 shaped
    like q: bf16(fp32(code * scale))."""
    if q.dtype != torch.uint8 or not q.is_cuda or not q.is_contiguous() or q.shape[-2:] != (
            N_KV_HEADS, HEAD_DIM):
        raise ValueError("q must be a contiguous uint8 CUDA tensor ending in [2, 256]")
    if (scale.dtype != torch.float32 or not scale.is_contiguous() or
            scale.shape != q.shape[:-1]):
        raise ValueError("scale must be a contiguous float32 tensor shaped like q[..., 0]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _bf16_cuda("out", out, q.shape)
    n_tok = q.numel() // (N_KV_HEADS * HEAD_DIM)
    _check(lib().ga_kv_dequantize_e4m3(_ptr(q), _ptr(scale), n_tok, _ptr(out), _stream()),
           "ga_kv_dequantize_e4m3")
    return out


def ga_prefill_e4m3_workspace_bytes(T: int) -> int:
    return lib().ga_prefill_e4m3_workspace_bytes(T)


def ga_attn_prefill_e4m3(qg, k_codes, k_scale, v_codes, v_scale, w_q, cos_tab, sin_tab,
                         q_base=0, T=None, causal=True, out=None, row_stats=None,
                         workspace=None):
    """ga_attn_prefill over e4m3 caches: k_codes, v_codes uint8 [T, 2, 256], k_scale,
    v_scale fp32 [T, 2] (as ga_kv_quantize_e4m3 writes them)."""
    rows = qg.shape[0]
    T = k_codes.shape[0] if T is None else T
    for n, t, dt in (("k_codes", k_codes, torch.uint8), ("v_codes", v_codes, torch.uint8),
                     ("k_scale", k_scale, torch.float32), ("v_scale", v_scale, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.shape[0] < T:
            raise ValueError(f"{n} must be a contiguous {dt} CUDA tensor with >= T rows")
    if out is None:
        out = torch.empty(rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=qg.device)
    if workspace is None:
        workspace = torch.empty(max(ga_prefill_e4m3_workspace_bytes(T), 1), dtype=torch.uint8,
                                device=qg.device)
    for n, t in (("qg", qg), ("w_q", w_q), ("cos_tab", cos_tab), ("sin_tab", sin_tab),
                 ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_prefill_e4m3(_ptr(qg), _ptr(k_codes), _ptr(k_scale), _ptr(v_codes),
                                      _ptr(v_scale), _ptr(w_q), _ptr(cos_tab), _ptr(sin_tab),
                                      cos_tab.shape[0], rows, T, q_base, 1 if causal else 0,
                                      _ptr(out), _ptr(row_stats), _ptr(workspace),
                                      workspace.numel(), _stream()),
           "ga_attn_prefill_e4m3")
    return out


def ga_attn_verify_e4m3(qg, k_codes, k_scale, v_codes, v_scale, seq_len, w_q, cos_tab, sin_tab,
                        out=None, workspace=None):
    """qg [n_seq, rows, 24, 512]; k_codes, v_codes uint8 [n_seq, cap, 2, 256]; k_scale,
    v_scale fp32 [n_seq, cap, 2] (as ga_kv_quantize_e4m3 writes them); seq_len: ints."""
    n_seq, rows = qg.shape[0], qg.shape[1]
    cap = k_codes.shape[1]
    for n, t, dt in (("k_codes", k_codes, torch.uint8), ("v_codes", v_codes, torch.uint8),
                     ("k_scale", k_scale, torch.float32), ("v_scale", v_scale, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.shape[:2] != (n_seq, cap):
            raise ValueError(f"{n} must be a contiguous {dt} CUDA tensor [n_seq, cap, ...]")
    lens = (ctypes.c_int * n_seq)(*[int(x) for x in seq_len])
    dev = qg.device
    if out is None:
        out = torch.empty(n_seq, rows, N_Q_HEADS * HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws_bytes = ga_verify_workspace_bytes(n_seq, rows, max(int(x) for x in seq_len))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    for n, t in (("qg", qg), ("w_q", w_q), ("cos_tab", cos_tab), ("sin_tab", sin_tab),
                 ("out", out)):
        _bf16_cuda(n, t)
    _check(lib().ga_attn_verify_e4m3(_ptr(qg), _ptr(k_codes), _ptr(k_scale), _ptr(v_codes),
                                     _ptr(v_scale), cap, lens, n_seq, rows, _ptr(w_q),
                                     _ptr(cos_tab), _ptr(sin_tab), cos_tab.shape[0], _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream()),
           "ga_attn_verify_e4m3")
    return out
