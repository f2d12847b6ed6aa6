"""Shared helpers of the GPU parity tests: seeded inputs on both sides, the library's
calls, the oracle's, and the element-wise comparison the tolerance is stated in.

Tolerance (the stated parity bar): |gpu - oracle| <= 2 bf16 ulp(oracle) + 1e-5 for every
element of outputs and weights, with ulp(x) = 2^(floor(log2|x|) - 7); the fraction of
elements more than 1 ulp away is reported as well.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import ga_oracle as O
from verify_gated_gqa_gb300 import binding as B
from verify_gated_gqa_gb300 import synth

SEED = 20261101


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def compare(got, want, n_ulp=2.0, atol=1e-5):
    g = np64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    ulp = O.ulp_bf16(w)
    err = np.abs(g - w)
    ok = err <= n_ulp * ulp + atol
    return {
        "n": int(w.size),
        "bad": int((~ok).sum()),
        "over_1ulp": float((err > ulp).mean()),
        "max_ulp": float(np.max(err / ulp)) if w.size else 0.0,
        "nan": int(np.isnan(g).sum()),
    }


# Every parity check of the session, in order: tests/conftest.py prints them as a table
# at the end of the run (so the record survives pytest's captured output and -q).
RECORDS = []


def _record(what, st, pairs=None, off=0, explained=0, passed=True):
    RECORDS.append({"what": what, "n": st["n"], "bad": st["bad"], "over_1ulp": st["over_1ulp"],
                    "max_ulp": st["max_ulp"], "pairs": pairs, "off": off,
                    "explained": explained, "passed": passed})


def assert_parity(got, want, what=""):
    st = compare(got, want)
    print(f"[parity] {what}: {st}")
    ok = st["nan"] == 0 and st["bad"] == 0
    _record(what, st, passed=ok)
    assert ok, f"{what}: {st}"
    return st


class Inputs:
    """One seeded problem: rows of fused q|gate at positions q_base.., T keys."""

    def __init__(self, seed, rows, T, device="cuda"):
        qg, k, v, w_q, w_k = synth.attention_inputs(seed, rows, T)
        self.cpu = dict(qg=qg, k=k, v=v, w_q=w_q, w_k=w_k)
        self.np = {n: np64(t) for n, t in self.cpu.items()}
        self.rows, self.T = rows, T
        self.device = device
        self._dev = None

    def dev(self):
        if self._dev is None:
            d = {n: t.to(self.device) for n, t in self.cpu.items()}
            n_pos = max(self.T, self.rows) + 16
            c, s = B.ga_rope_table_host(n_pos)
            d["cos"], d["sin"] = c.to(self.device), s.to(self.device)
            d["k_prep"] = B.ga_k_prologue(d["k"], d["w_k"], d["cos"], d["sin"])
            self._dev = d
        return self._dev

    def oracle_tables(self, mode="R1"):
        n_pos = max(self.T, self.rows) + 16
        return O.rope_tables(n_pos, rounded=(mode != "F64"))

    def oracle_keys(self, mode="R1"):
        if getattr(self, "_okeys", None) is None:
            c, s = self.oracle_tables(mode)
            self._okeys = O.prep_keys(self.np["k"], self.np["w_k"], c, s, mode=mode)
        return self._okeys

    def ref(self, q_base, T, kind, rows=None, heads=None, mask=None, qg=None,
            want_weights=False):
        """AttnRef of this problem (qg defaults to all rows; pass the window's rows)."""
        c, s = self.oracle_tables()
        return AttnRef(self.np["qg"] if qg is None else qg, self.oracle_keys(), self.np["v"],
                       self.np["w_q"], c, s, q_base, T, kind, mask, rows, heads, want_weights)


# ------------------------------------------------------------------ ambiguous roundings
# The score is "the bf16 GEMM result rounded" (pegainfer PR #1151, the commit that adds the
# attention reader), and "the float32 reduction order is this kernel's own". When the
# exact dot product lies within the fp32 reduction error of a bf16 rounding midpoint,
# either neighbour is a correct score. The band below is the tensor core's measured
# accumulation error (at most 8.3 fp32 ulps of the largest 16-product prefix sum over
# 2^20 dot products of normalised bf16 rows), doubled. Likewise the exponential is
# evaluated in fp32 (argument rounding plus ex2.approx, <= 2.06 ulps exhaustively over
# [-32, 8]); a weight whose exact value lies inside that band of a midpoint may take
# either neighbour. A (row, head) that misses the tolerance against the oracle passes only
# if some choice of neighbours for its ambiguous roundings reproduces the GPU row (all 256
# outputs, and the weights when given) within the same tolerance.
TC_BAND_ULP32 = 16.0
MAX_ALTERNATIVES = 10
# At most this fraction of a check's (row, head) pairs may miss the tolerance and still be
# explained by ambiguous roundings (never fewer than MIN_OFF_CAP pairs); beyond it the check
# fails without a search. Calibration (every GPU parity check of the suite on GB300): the
# explained pairs were 0.26 % of all pairs checked, at most 0.42 % in a check of more than
# 10,000 pairs (S = 2048 bidirectional) and at most 5 pairs in a check of fewer than 1,000
# (S = 8192 sampled rows, 768 pairs): the cap is about 2.4 times the largest large-sample
# rate, with a floor for the small samples.
MAX_OFF_FRACTION = 0.01
MIN_OFF_CAP = 8


def off_cap(pairs):
    return max(MIN_OFF_CAP, int(np.ceil(MAX_OFF_FRACTION * pairs)))


def _ulp32(x):
    x = np.abs(np.asarray(x, np.float64))
    m, e = np.frexp(np.where(x > 0, x, 1.0))
    return np.where(x > 0, np.ldexp(1.0, e - 24), 2.0 ** -149)


def _alternatives(q, kk, band_fn_exp):
    """Per visible key: exact dot, the oracle's bf16 score, and an alternative bf16 score
    (nan if the rounding is not ambiguous)."""
    prods = q[None, :] * kk                          # exact products
    pref = np.cumsum(prods.reshape(len(kk), 16, 16).sum(axis=2), axis=1)
    band = TC_BAND_ULP32 * _ulp32(np.max(np.abs(pref), axis=1))
    dot = prods.sum(axis=1)
    b = O.bf16(dot)
    up, dn = O.bf16(dot + band), O.bf16(dot - band)
    alt = np.where(up != b, up, np.where(dn != b, dn, np.nan))
    return dot, b, alt


class AttnRef:
    """Oracle results for selected rows/heads plus what the ambiguity analysis needs."""

    def __init__(self, qg, k_hat, v, w_q, cos, sin, q_base, T, kind, mask=None, rows=None,
                 heads=None, want_weights=False):
        qg = np.asarray(qg, np.float64)
        self.rows = np.arange(qg.shape[0]) if rows is None else np.asarray(rows)
        self.heads = list(range(24)) if heads is None else list(heads)
        self.q_hat, self.gate = O.prep_queries(qg, w_q, cos, sin, q_base, rows=self.rows)
        self.k_hat = np.asarray(k_hat, np.float64)[:T]
        self.v = np.asarray(v, np.float64)[:T]
        self.vis = O.visibility(kind, self.rows, T, q_base, mask)
        self.out, self.weights, self.hidden = O.attention(
            self.q_hat, self.gate, self.k_hat, self.v, self.vis, heads=self.heads,
            want_weights=want_weights)

    def cols(self):
        return np.concatenate([np.arange(h * 256, (h + 1) * 256) for h in self.heads])

    def _explain(self, i, h, got_o, got_w):
        kv = h // 12
        vis = self.vis[i]
        idx = np.nonzero(vis)[0]
        q = self.q_hat[i, h]
        kk = self.k_hat[idx, kv]
        vv = self.v[idx, kv]
        dot, b, alt_s = _alternatives(q, kk, None)
        s = b / 16.0
        w_hat = O.bf16_sig(np.exp(s))
        t = s * np.log2(np.e)
        rel = np.log(2) * 3 * max(np.max(np.abs(t)), 1.0) * 2.0 ** -24 + 2.1 * 2.0 ** -23
        w_up, w_dn = O.bf16_sig(np.exp(s) * (1 + rel)), O.bf16_sig(np.exp(s) * (1 - rel))
        alt_w = np.where(w_up != w_hat, w_up, np.where(w_dn != w_hat, w_dn, np.nan))
        # candidate changes of single weights: alternative score, alternative exponential
        cand = []
        for j in np.nonzero(~np.isnan(alt_s))[0]:
            cand.append((j, O.bf16_sig(np.exp(alt_s[j] / 16.0)) - w_hat[j]))
        for j in np.nonzero(~np.isnan(alt_w))[0]:
            cand.append((j, alt_w[j] - w_hat[j]))
        if not cand:
            return False
        cand.sort(key=lambda c: -abs(c[1]) * np.abs(vv[c[0]]).max())
        cand = cand[:MAX_ALTERNATIVES]
        g = O.sigmoid_gate(self.gate[i, h])
        L0 = w_hat.sum()
        num0 = w_hat @ vv
        n = len(cand)
        for mask in range(1, 1 << n):
            dw = np.zeros(len(idx))
            for c in range(n):
                if mask >> c & 1:
                    dw[cand[c][0]] += cand[c][1]
            L = L0 + dw.sum()
            o = O.bf16((num0 + dw @ vv) / L)
            out = O.bf16(o * g)
            if not np.all(O.within_tolerance(got_o, out)):
                continue
            if got_w is not None:
                w_row = np.zeros(self.vis.shape[1])
                w_row[idx] = O.bf16((w_hat + dw) / L)
                if not np.all(O.within_tolerance(got_w, w_row)):
                    continue
            return True
        return False

    def check(self, got_out, got_weights=None, what=""):
        """got_out [len(rows), 6144] (GPU); got_weights [24, len(rows), T] or None."""
        cols = self.cols()
        g = np64(got_out)[:, cols]
        w = self.out[:, cols]
        st = compare(g, w)
        ok = O.within_tolerance(g, w) & ~np.isnan(g)
        gw = None
        bad_pairs = set()
        for i, c in zip(*np.nonzero(~ok)):
            bad_pairs.add((int(i), self.heads[c // 256]))
        if got_weights is not None:
            gw = np64(got_weights)
            stw = compare(gw[self.heads], self.weights[self.heads])
            okw = O.within_tolerance(gw[self.heads], self.weights[self.heads])
            for hh, i, _ in zip(*np.nonzero(~okw)):
                bad_pairs.add((int(i), self.heads[hh]))
            st["weights"] = stw
        unexplained = []
        pairs = len(self.rows) * len(self.heads)
        if len(bad_pairs) > off_cap(pairs):
            # far more rows off than rounding ties produce: a real error, report it at once
            st["rows_off_oracle"] = len(bad_pairs)
            print(f"[parity] {what}: {st}")
            _record(what, st, pairs, len(bad_pairs), 0, False)
            raise AssertionError(f"{what}: {len(bad_pairs)} of {pairs} (row, head) pairs off "
                                 f"the oracle, above the cap {off_cap(pairs)}: {st}")
        for i, h in sorted(bad_pairs):
            go = np64(got_out)[i, h * 256:(h + 1) * 256]
            gwr = None if gw is None else gw[h, i]
            if not self._explain(i, h, go, gwr):
                unexplained.append((int(self.rows[i]), h))
        st["rows_off_oracle"] = len(bad_pairs)
        st["explained_by_ambiguous_rounding"] = len(bad_pairs) - len(unexplained)
        st["unexplained"] = unexplained[:10]
        print(f"[parity] {what}: {st}")
        ok = st["nan"] == 0 and not unexplained
        _record(what, st, pairs, len(bad_pairs), st["explained_by_ambiguous_rounding"], ok)
        assert ok, f"{what}: {st}"
        return st
