"""The multi-GPU split of a pass (KV-head groups, then causal row windows), run as gloo ranks
on the CPU with the oracle standing in for each GPU: every rank computes its share (its KV
heads' query heads over its row window, a window call at its own q_base), the shares are
summed across ranks (they are disjoint, so the sum only assembles them), and the result is
the full oracle pass exactly; every (row, head) output is covered once."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

S = 200
SEED = 20261101 + 70


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from oracle import ga_oracle as O
    from verify_gated_gqa_gb300 import synth
    qg, k, v, w_q, w_k = (t.double().numpy() for t in synth.attention_inputs(SEED, S, S))
    c, s = O.rope_tables(S)
    return qg, O.prep_keys(k, w_k, c, s), v, w_q, c, s


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import ga_oracle as O
    from verify_gated_gqa_gb300 import shard
    qg, kp, v, w_q, c, s = _inputs()
    sh = shard.plan(world, S)[rank]
    part = np.zeros((S, 24 * 256))
    cover = np.zeros((S, 24))
    r0, n = sh["row0"], sh["rows"]
    heads = list(shard.heads_of(sh))
    if n:
        part[r0:r0 + n] = O.prefill(qg[r0:r0 + n], kp, v, w_q, c, s, r0, r0 + n, True,
                                    heads=heads)
        cover[r0:r0 + n, heads] = 1
    t_part, t_cover = torch.from_numpy(part), torch.from_numpy(cover)
    torch.distributed.all_reduce(t_part)
    torch.distributed.all_reduce(t_cover)
    if rank == 0:
        full = O.prefill(qg, kp, v, w_q, c, s, 0, S, True)
        results["equal"] = bool(np.array_equal(t_part.numpy(), full))
        results["covered_once"] = bool(np.all(t_cover.numpy() == 1))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_split_shares_assemble_the_full_pass(world):
    port = _free_port()
    results = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True,
                       start_method="spawn")
    assert results["equal"] and results["covered_once"]


def test_plan_covers_rows_and_heads_once():
    from verify_gated_gqa_gb300 import shard
    for world in range(1, 9):
        for rows in (1, 64, 200, 8192):
            cover = np.zeros((rows, 24), int)
            for sh in shard.plan(world, rows):
                assert sh["row0"] % shard.ROW_ALIGN == 0 or sh["rows"] == 0
                cover[sh["row0"]:sh["row0"] + sh["rows"], list(shard.heads_of(sh))] += 1
            assert np.all(cover == 1), (world, rows)
    # causal windows balance the visible pairs: at S = 8192 over 4 windows each share is
    # within one 64-row step of a quarter
    w = shard.row_windows(8192, 4)
    work = [shard._pairs(r0, r0 + n, 0, 8192, True) for r0, n in w]
    assert max(work) / min(work) < 1.1
