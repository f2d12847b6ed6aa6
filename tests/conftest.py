import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built library")
    config.addinivalue_line("markers", "slow: long CPU-only test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One line per parity check of the session against the oracle: elements compared,
    elements outside 2 bf16 ulp + 1e-5 ('bad'), the fraction over 1 ulp, the largest error
    in ulps, and the (row, head) pairs off the oracle with how many of them the ambiguous-
    rounding rule explained (tests/parity.py). Checks that must fail are marked."""
    mod = sys.modules.get("tests.parity")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the oracle (tolerance 2 bf16 ulp + 1e-5 per element)")
    tr.write_line("check | elements | bad | over 1 ulp | max ulp | pairs off/checked (cap) | "
                  "explained | result")
    # the named configurations last, so that the end of the log always holds them
    named = ("S=64 causal", "S=2048 causal", "S=2048 bidirectional", "S=8192 causal",
             "S=8192 chunk", "masked S=8192", "verify 8 x 16")
    key = lambda r: any(r["what"].startswith(n) for n in named)
    recs = [r for r in recs if not key(r)] + [r for r in recs if key(r)]
    for r in recs:
        pairs = r["pairs"]
        po = (f"{r['off']}/{pairs} ({mod.off_cap(pairs)})" if pairs else "-")
        tr.write_line(f"{r['what']} | {r['n']} | {r['bad']} | {r['over_1ulp']:.2e} | "
                      f"{r['max_ulp']:.2f} | {po} | {r['explained']} | "
                      f"{'pass' if r['passed'] else 'FAIL'}")
