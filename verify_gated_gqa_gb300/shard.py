"""How one causal, bidirectional or stored-mask pass splits over GPUs with no exchange
between them.

Query head h reads only KV head h // 12, so each KV head with its 12 query heads is an
independent problem (ga_attn_prefill_kv / ga_attn_masked_kv run one group and write only
its output columns). Query rows are independent too once a GPU holds the keys and values
they attend to, so a group's rows can be cut further into windows (each window a call at
its own q_base, a multiple of 64). A rank's share is therefore (KV-head group, row window);
the shares cover every (row, head) output exactly once and need no collective: gathering
the output columns and rows is the caller's business.

This module only plans; it computes nothing of the attention.
"""
from __future__ import annotations

N_KV_HEADS = 2
GROUP = 12            # query heads per KV head
ROW_ALIGN = 64        # a window's first row (its q_base offset) is a multiple of 64


def _pairs(r0: int, r1: int, q_base: int, T: int, causal: bool) -> int:
    """Visible (query, key) pairs of rows r0 .. r1-1 (row r at position q_base + r)."""
    if not causal:
        return (r1 - r0) * T
    a, b = q_base + r0 + 1, q_base + r1
    return (a + b) * (r1 - r0) // 2


def row_windows(rows: int, n: int, q_base: int = 0, T: int | None = None,
                causal: bool = True) -> list[tuple[int, int]]:
    """n contiguous windows (row0, nrows) covering rows 0 .. rows-1, each starting at a
    multiple of ROW_ALIGN, cut where the running count of visible pairs crosses k/n of the
    total (so causal windows get about equal work). Windows may be empty."""
    if n < 1:
        raise ValueError("n >= 1")
    T = q_base + rows if T is None else T
    total = _pairs(0, rows, q_base, T, causal)
    candidates = list(range(0, rows, ROW_ALIGN)) + [rows]
    cuts = [0]
    for k in range(1, n):
        target = total * k / n
        c = next((c for c in candidates if c >= cuts[-1] and _pairs(0, c, q_base, T, causal)
                  >= target), rows)
        cuts.append(c)
    cuts.append(rows)
    return [(cuts[i], cuts[i + 1] - cuts[i]) for i in range(n)]


def plan(world: int, rows: int, q_base: int = 0, T: int | None = None,
         causal: bool = True) -> list[dict]:
    """Each rank's share of one pass: {"kv_first", "kv_count", "row0", "rows"}. An even
    world splits the two KV-head groups first (half the ranks each) and then rows; an odd
    world splits rows only (every rank runs both groups)."""
    if world < 1:
        raise ValueError("world >= 1")
    kv_split = N_KV_HEADS if world % N_KV_HEADS == 0 else 1
    per_group = world // kv_split
    windows = row_windows(rows, per_group, q_base, T, causal)
    shares = []
    for rank in range(world):
        g, w = divmod(rank, per_group)
        kv_count = N_KV_HEADS // kv_split
        row0, nrows = windows[w]
        shares.append({"kv_first": g * kv_count, "kv_count": kv_count, "row0": row0,
                       "rows": nrows})
    return shares


def heads_of(share: dict) -> range:
    """The query heads a share computes."""
    return range(GROUP * share["kv_first"], GROUP * (share["kv_first"] + share["kv_count"]))
