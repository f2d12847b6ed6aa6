"""Benchmark of the gated GQA attention hot path on GB300.

Workload (one step): long causal prefill at S = 8192, batch 1, 24 query heads over 2 KV
heads, head_dim 256, 64-dim partial RoPE, (1+w) RMSNorm: the K prologue over all 8192
keys, the Q prologue over all 8192 x 24 query rows, then the full causal pass (Q.K^T,
online softmax, P.V, gated epilogue). The step runs both prologues in one launch
(ga_qk_prologue; --prologues side or serial runs them as two) and then
ga_attn_prefill_prepared, so that the prologues and the attention are each timed alone.
Inputs are seeded synthetic bf16 N(0,1) activations and N(0,0.1) norm weights.

Metric: algorithmic TFLOP/s, 4 * head_dim * heads per visible (query, key) pair (the
convention under which pegainfer PR #1151's 2048 x 2048 table gives 0.93 TFLOP/s);
tokens/s is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs one independent sequence per GPU (weak scaling; no data-path collective:
the process group only carries the barrier and the max-over-ranks time).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

S = 8192
HEADS, KV_HEADS, DIM = 24, 2, 256
SEED = 20261101 + 3
METRIC = "causal prefill attention TFLOP/s at S=8192 (tokens/s beside)"
UNIT = "TFLOP/s"
WORKLOAD = "causal gated GQA prefill, batch 1, S=8192, 24q/2kv heads, d=256, rope 64/256"


def visible_pairs_causal(rows: int, T: int, q_base: int = 0) -> int:
    """Sum over rows of the keys a causal row sees (row r sees q_base + r + 1 keys)."""
    first = q_base + 1
    last = q_base + rows
    return (first + last) * rows // 2


def attention_flops(pairs: int) -> float:
    return 4.0 * DIM * HEADS * pairs


FLOPS_STEP = attention_flops(visible_pairs_causal(S, S))  # 824.73 GFLOP


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, max clock, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], r[5:9]):
                if v.strip().lower() in ("active", "1", "yes"):
                    reasons.add(n)
        loaded = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- the GPU arm
def make_inputs(device, seed):
    from verify_gated_gqa_gb300 import synth
    return synth.attention_inputs(seed, S, S, device=device)


def run_gpu(args, world, rank, local):
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    qg, k, v, w_q, w_k = make_inputs(dev, SEED + rank)
    c, s = B.ga_rope_table_host(S)
    cos, sin = c.to(dev), s.to(dev)
    k_prep = torch.empty_like(k)
    out = torch.empty(S, HEADS * DIM, dtype=torch.bfloat16, device=dev)

    q_prep = out.view(S, HEADS, DIM)   # as in ga_attn_prefill: the output buffer holds Q first
    joint = args.prologues == "joint"

    def step():
        if joint:
            B.ga_qk_prologue(k, w_k, qg, w_q, cos, sin, k_prep=k_prep, q_prep=q_prep)
        else:
            B.ga_k_prologue(k, w_k, cos, sin, k_prep=k_prep)
            B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)
        B.ga_attn_prefill_prepared(out, qg, k_prep, v, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # device-timed region: K back-to-back steps; per-kernel events on the same stream
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # --prologues joint (the default): both prologues in one launch (ga_qk_prologue);
    # side: the key prologue on a side stream beside the query prologue, after the previous
    # step's attention has read k_prep, the attention waiting for both; serial: all three
    # on one stream.
    side = torch.cuda.Stream(device=dev)
    k_done = [torch.cuda.Event() for _ in range(args.steps)]
    serial, side_mode = args.prologues == "serial", args.prologues == "side"
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        if joint:
            B.ga_qk_prologue(k, w_k, qg, w_q, cos, sin, k_prep=k_prep, q_prep=q_prep)
            ev[i][1].record(stream)
        elif serial:
            B.ga_k_prologue(k, w_k, cos, sin, k_prep=k_prep)
            ev[i][1].record(stream)
        else:
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                B.ga_k_prologue(k, w_k, cos, sin, k_prep=k_prep)
                ev[i][1].record(side)
                k_done[i].record(side)
        if not joint:
            B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)
        ev[i][2].record(stream)
        if side_mode:
            stream.wait_event(k_done[i])
        B.ga_attn_prefill_prepared(out, qg, k_prep, v, out=out)
        ev[i][3].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = total_ms / args.steps
    pro_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps))
    qpro_ms = statistics.mean((ev[i][1] if serial else ev[i][0]).elapsed_time(
        ev[i][2]) for i in range(args.steps))
    attn_ms = statistics.mean(ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps))
    status = B.ga_device_status()

    # end to end through the C ABI with host buffers: every step copies its inputs from
    # pinned host memory (H2D), runs the two public calls (ga_k_prologue, ga_attn_prefill)
    # and reads its output back into pinned host memory (D2H). Steps are pipelined on three
    # streams with double-buffered device inputs and outputs, as a serving loop would run
    # them: step i+1's inputs travel while step i computes and step i-1's output returns.
    host_in = [t.cpu().pin_memory() for t in (qg, k, v, w_q, w_k, cos, sin)]

    def compute(d, o):
        qg_d, k_d, v_d, wq_d, wk_d, cos_d, sin_d = d
        if joint:
            B.ga_qk_prologue(k_d, wk_d, qg_d, wq_d, cos_d, sin_d, k_prep=k_prep,
                             q_prep=o.view(S, HEADS, DIM))
            B.ga_attn_prefill_prepared(o, qg_d, k_prep, v_d, out=o)
        else:
            B.ga_k_prologue(k_d, wk_d, cos_d, sin_d, k_prep=k_prep)
            B.ga_attn_prefill(qg_d, k_prep, v_d, wq_d, cos_d, sin_d, 0, S, out=o)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = e2e_pipelined(host_in, compute, out, e2e_steps, world, dev)
    secondary = (None if args.no_secondary else
                 secondary_measurements(dev, rank, max(3, min(args.steps, 20))))

    if rank != 0:
        return None
    peak_tf, peak_hbm, peak_src = measured_peaks()
    achieved = FLOPS_STEP / (attn_ms * 1e-3) / 1e12
    value = world * FLOPS_STEP / (ms_step * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": S,
                   "parallelism": f"independent sequence per GPU x{world}",
                   "l2": "inputs larger than L2 (qg 192 MiB read + out 96 MiB written per step)",
                   "step": (("ga_qk_prologue (8192 keys and 8192 x 24 query rows in one "
                             "launch)" if joint else
                             "ga_k_prologue (8192 keys) + ga_q_prologue (8192 x 24 rows)")
                            + " + ga_attn_prefill_prepared (8192 rows, causal)"
                            + ("; the key prologue on a side stream beside the query "
                               "prologue, joined before the attention" if side_mode else ""))},
        "tokens_per_s": round(world * S / (ms_step * 1e-3), 1),
        "kernel_ms": ({"attn_kernel": round(attn_ms, 4), "qk_prologue": round(pro_ms, 4)}
                      if joint else
                      {"attn_kernel": round(attn_ms, 4), "k_prologue": round(pro_ms, 4),
                       "q_prologue": round(qpro_ms, 4),
                       "prologues": "serial" if serial else
                                    "concurrent (each span includes the other's overlap)"}),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "traffic": ATTN_TRAFFIC_BYTES,
                     "peak_kind": f"dense bf16 burst ({peak_src})",
                     "kernel": "attn_kernel", "algorithmic_flops": FLOPS_STEP},
        "e2e": {"value": round(world * FLOPS_STEP / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "schedule": "H2D, compute ("
                            + ("ga_qk_prologue + ga_attn_prefill_prepared" if joint else
                               "ga_k_prologue + ga_attn_prefill")
                            + ") and D2H on three streams, device inputs and outputs "
                              "double-buffered"},
        "gpu_launches": (2 if joint else 3) * args.steps,
        "clocks": clk,
        "device_status": status,
        "secondary": secondary,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, gpu_out=out)
    return line


def e2e_pipelined(host_in, compute, out, n, world, dev):
    """End to end through the C ABI with host buffers: every step copies its inputs from
    pinned host memory (H2D), runs `compute(device inputs, device output)` (the public
    calls) and reads its output back into pinned host memory (D2H). Steps are pipelined on
    three streams with double-buffered device inputs and outputs, as a serving loop would
    run them: step i+1's inputs travel while step i computes and step i-1's output returns.
    Returns (ms per step, max over ranks; H2D bytes per step; D2H bytes per step)."""
    stream = torch.cuda.current_stream()
    dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h_stream, c_stream, d_stream = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        h_done = [torch.cuda.Event() for _ in range(n)]
        c_done = [torch.cuda.Event() for _ in range(n)]
        d_done = [torch.cuda.Event() for _ in range(n)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h_stream.wait_event(start)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(h_stream):
                if i >= 2:
                    h_stream.wait_event(c_done[i - 2])   # buffer b's inputs are consumed
                for h, d in zip(host_in, dev_in[b]):
                    d.copy_(h, non_blocking=True)
                h_done[i].record(h_stream)
            with torch.cuda.stream(c_stream):
                c_stream.wait_event(h_done[i])
                if i >= 2:
                    c_stream.wait_event(d_done[i - 2])   # buffer b's output was read back
                compute(dev_in[b], outs[b])
                c_done[i].record(c_stream)
            with torch.cuda.stream(d_stream):
                d_stream.wait_event(c_done[i])
                host_out[b].copy_(outs[b], non_blocking=True)
                d_done[i].record(d_stream)
        stream.wait_event(d_done[n - 1])
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run(2)
    barrier(world)
    ms = max_over_ranks(run(n), world, dev) / n
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    return ms, h2d, d2h


# ---------------------------------------------------------------- verify windows (8 x 16 rows, L = 65,536)
V_ROWS, V_L = 16, 65536
V_CAP = V_L + V_ROWS
V_PAGE = 256   # positions per page of the paged-cache workload


def verify_bytes(n_seq):
    return (2 * n_seq * V_CAP * KV_HEADS * DIM * 2       # K and V caches, read once
            + n_seq * V_ROWS * HEADS * 2 * DIM * 2     # fused q|gate rows
            + n_seq * V_ROWS * HEADS * DIM * 2)        # output rows


def verify_setup(dev, seed, n_seq, paged=False, e4m3=False):
    """Prepared K/V caches of n_seq sequences (65,552 positions each) resident in HBM, the
    fused rows of their 16 new rows, and one step: the verify call over them. Returns
    (step, algorithmic bytes per step)."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300 import synth
    c, s = B.ga_rope_table_host(V_CAP)
    cos, sin = c.to(dev), s.to(dev)
    w_q = synth.normal_bf16(seed, "w_q", (DIM,), sigma=0.1, device=dev)
    w_k = synth.normal_bf16(seed, "w_k", (DIM,), sigma=0.1, device=dev)
    k_cache = torch.empty(n_seq, V_CAP, KV_HEADS, DIM, dtype=torch.bfloat16, device=dev)
    v_cache = torch.empty_like(k_cache)
    for b in range(n_seq):
        k_raw = synth.normal_bf16(seed, "k", (V_CAP, KV_HEADS, DIM), sub=b, device=dev)
        B.ga_k_prologue(k_raw, w_k, cos, sin, k_prep=k_cache[b])
        v_cache[b] = synth.normal_bf16(seed, "v", (V_CAP, KV_HEADS, DIM), sub=b, device=dev)
        del k_raw
    qg = torch.stack([synth.normal_bf16(seed, "qg", (V_ROWS, HEADS, 2 * DIM), sub=b, device=dev)
                      for b in range(n_seq)])
    lens = [V_L] * n_seq
    out = torch.empty(n_seq, V_ROWS, HEADS * DIM, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.ga_verify_workspace_bytes(n_seq, V_ROWS, V_L), dtype=torch.uint8,
                     device=dev)
    n_bytes = verify_bytes(n_seq)
    if e4m3:
        # the same caches as e4m3 rows with an fp32 scale each (algorithmic bytes: the codes
        # and scales read once, the fused rows and the outputs)
        k8, ksc = B.ga_kv_quantize_e4m3(k_cache)
        v8, vsc = B.ga_kv_quantize_e4m3(v_cache)
        del k_cache, v_cache
        n_bytes = (k8.numel() + v8.numel() + 4 * (ksc.numel() + vsc.numel())
                   + qg.numel() * 2 + out.numel() * 2)

        def step():
            B.ga_attn_verify_e4m3(qg, k8, ksc, v8, vsc, lens, w_q, cos, sin, out=out, workspace=ws)
    elif paged:
        pages_per_seq = -(-V_CAP // V_PAGE)
        n_pages = n_seq * pages_per_seq
        order = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
        table = order.view(n_seq, pages_per_seq).to(torch.int32).to(dev)
        k_pool = torch.zeros(n_pages, V_PAGE, KV_HEADS, DIM, dtype=torch.bfloat16, device=dev)
        v_pool = torch.zeros_like(k_pool)
        for b in range(n_seq):
            for p in range(pages_per_seq):
                lo, hi = p * V_PAGE, min((p + 1) * V_PAGE, V_CAP)
                pg = int(order[b * pages_per_seq + p])
                k_pool[pg, :hi - lo] = k_cache[b, lo:hi]
                v_pool[pg, :hi - lo] = v_cache[b, lo:hi]
        del k_cache, v_cache

        def step():
            B.ga_attn_verify_paged(qg, k_pool, v_pool, table, lens, w_q, cos, sin, out=out,
                                   workspace=ws)
    else:
        def step():
            B.ga_attn_verify(qg, k_cache, v_cache, lens, w_q, cos, sin, out=out, workspace=ws)
    return step, n_bytes


def timed_steps(step, steps, warmup, stream):
    """ms per step of `steps` back-to-back steps after `warmup` untimed ones (CUDA events
    on the launching stream, synchronised on both sides)."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def run_verify(args, world, rank, local):
    """Verify windows on one GPU (per rank): ga_attn_verify over prepared caches resident in
    HBM, 16 rows over 65,536 cached keys per sequence (--verify-seqs sequences; 8 is the
    workload, fewer only for profiling). With
    --workload verify_paged the same caches sit in pages of 256 positions scattered over
    two page pools in a seeded random order, read through ga_attn_verify_paged."""
    V_SEQ = args.verify_seqs
    paged = args.workload == "verify_paged"
    e4m3 = args.workload == "verify_e4m3"
    kind = " over paged caches" if paged else (" over e4m3 caches" if e4m3 else "")
    V_METRIC = (f"verify windows{kind}: HBM GB/s ({V_SEQ} sequences x 16 rows over L=65536 "
                "cached keys)")
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    step, V_BYTES = verify_setup(dev, SEED + 5 + rank, V_SEQ, paged, e4m3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    if rank != 0:
        return None
    _, peak_hbm, peak_src = measured_peaks()
    gbs = V_BYTES / (ms * 1e-3) / 1e9
    return {
        "metric": V_METRIC, "value": round(world * gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": f"verify: {V_SEQ} sequences x 16 rows at positions 65536..65551 over "
                               "prepared K/V caches [65552, 2, 256] bf16, split-key partials "
                               "and combine" + (f"; caches in pages of {V_PAGE} positions, "
                                                "scattered over two page pools" if paged else "")
                               + ("; caches as e4m3 rows with an fp32 scale each (half the "
                                  "bytes), widened to bf16 in shared memory" if e4m3 else ""),
                   "l2": f"K/V caches {2 * V_SEQ * V_CAP * KV_HEADS * DIM * 2 / 1e9:.2f} GB"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                     "frac": round(gbs / peak_hbm, 4),
                     "traffic": (VERIFY_ATTN_TRAFFIC_BYTES if V_SEQ == 8 and not paged and not e4m3
                                 else None),
                     "traffic_kernel": "attn_kernel (verify variant), the call's dominant launch",
                     "peak_kind": f"HBM copy ({peak_src})",
                     "kernel": f"ga_attn_verify{'_paged' if paged else ('_e4m3' if e4m3 else '')} "
                               "(Q prologue + attn_kernel<verify> + combine)",
                     "algorithmic_bytes": V_BYTES},
        "gpu_launches": 3 * args.steps, "clocks": clk, "device_status": B.ga_device_status(),
    }


# ---------------------------------------------------------------- sparse-selection masked attention (S = 8192)
M_WINDOW, M_RANDOM = 128, 1024


def masked_setup(dev, seed):
    """The stored-mask workload at the 8192-token cap: seeded inputs, the selection mask
    (each row's causal window of 128 keys plus 1024 random earlier keys) resident in HBM,
    the prepared keys, and the counts of its work: visible (query, key) pairs and the
    128 x 128 tiles with a visible key (the tiles the kernel executes)."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300 import synth
    qg, kraw, v, w_q, w_k = synth.attention_inputs(seed, S, S, device=dev)
    mask = synth.selection_mask(seed, S, window=M_WINDOW, n_random=M_RANDOM, device=dev)
    c, s_ = B.ga_rope_table_host(S)
    cos, sin = c.to(dev), s_.to(dev)
    k_prep = B.ga_k_prologue(kraw, w_k, cos, sin)
    pairs = int(mask.sum(dtype=torch.int64).item())
    tiles = int((mask.view(S // 128, 128, S // 128, 128).amax(dim=(1, 3)) != 0).sum().item())
    return dict(qg=qg, kraw=kraw, v=v, w_q=w_q, w_k=w_k, mask=mask, cos=cos, sin=sin,
                k_prep=k_prep, pairs=pairs, flops=attention_flops(pairs),
                exec_flops=4.0 * DIM * HEADS * tiles * 128 * 128, tiles=tiles)


def run_masked(args, world, rank, local):
    """Sparse-selection masked attention at S = 8192: each step runs the key and query
    prologues (one ga_qk_prologue launch; with --prologues side or serial, ga_k_prologue then
    ga_q_prologue) and ga_attn_masked_prepared (the mask prepass and the attention), the
    pieces ga_attn_masked runs, each timed on the stream. TFLOP/s both on the algorithmic
    work (visible pairs) and on the executed 128 x 128 tiles."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    m = masked_setup(dev, SEED + 7 + rank)
    qg, kraw, v, w_q, w_k, mask, cos, sin = (m[n] for n in ("qg", "kraw", "v", "w_q", "w_k",
                                                             "mask", "cos", "sin"))
    k_prep = torch.empty_like(kraw)
    q_prep = torch.empty(S, HEADS, DIM, dtype=torch.bfloat16, device=dev)
    out = torch.empty(S, HEADS * DIM, dtype=torch.bfloat16, device=dev)
    hid = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(B.ga_masked_workspace_bytes(S, S), dtype=torch.uint8, device=dev)

    joint = args.prologues == "joint"

    def prologues():
        if joint:
            B.ga_qk_prologue(kraw, w_k, qg, w_q, cos, sin, k_prep=k_prep, q_prep=q_prep)
        else:
            B.ga_k_prologue(kraw, w_k, cos, sin, k_prep=k_prep)
            B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)

    def step():
        prologues()
        B.ga_attn_masked_prepared(q_prep, qg, k_prep, v, mask, out=out, hidden_rows=hid,
                                  workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        if joint:
            B.ga_qk_prologue(kraw, w_k, qg, w_q, cos, sin, k_prep=k_prep, q_prep=q_prep)
            ev[i][1].record(stream)
        else:
            B.ga_k_prologue(kraw, w_k, cos, sin, k_prep=k_prep)
            ev[i][1].record(stream)
            B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)
        ev[i][2].record(stream)
        B.ga_attn_masked_prepared(q_prep, qg, k_prep, v, mask, out=out, hidden_rows=hid,
                                  workspace=ws)
        ev[i][3].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    span = lambda a, b: statistics.mean(ev[i][a].elapsed_time(ev[i][b]) for i in range(args.steps))
    kpro_ms, qpro_ms, attn_ms = span(0, 1), span(1, 2), span(2, 3)
    status = B.ga_device_status()
    hidden = int(hid.item())

    host_in = [t.cpu().pin_memory() for t in (qg, kraw, v, w_q, w_k, cos, sin, mask)]
    ws2 = torch.empty_like(ws)

    def compute(d, o):
        qg_d, k_d, v_d, wq_d, wk_d, cos_d, sin_d, m_d = d
        B.ga_k_prologue(k_d, wk_d, cos_d, sin_d, k_prep=k_prep)
        B.ga_attn_masked(qg_d, k_prep, v_d, wq_d, cos_d, sin_d, m_d, out=o, hidden_rows=hid,
                         workspace=ws2)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = e2e_pipelined(host_in, compute, out, e2e_steps, world, dev)
    if rank != 0:
        return None
    peak_tf, _, peak_src = measured_peaks()
    flops, exec_flops = m["flops"], m["exec_flops"]
    achieved = flops / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": "sparse-selection masked attention TFLOP/s at S=8192 (algorithmic: visible "
                  "pairs)",
        "value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights, seeded selection "
                "mask)",
        "config": {"workload": f"masked gated GQA, S=8192 (the cap), 24q/2kv heads, d=256, "
                               f"stored uint8 mask [8192, 8192]: each row's causal window of "
                               f"{M_WINDOW} keys plus {M_RANDOM} random earlier keys",
                   "global_batch": world, "seq_len": S,
                   "parallelism": f"independent sequence per GPU x{world}",
                   "l2": "inputs larger than L2 (qg 192 MiB + mask 64 MiB read, out 96 MiB "
                         "written per step)",
                   "step": ("ga_qk_prologue (both prologues, one launch)" if joint else
                            "ga_k_prologue + ga_q_prologue")
                           + " + ga_attn_masked_prepared (mask prepass + attention), the "
                             "pieces of ga_attn_masked"},
        "visible_pairs_per_head": m["pairs"], "algorithmic_gflop": round(flops / 1e9, 2),
        "executed_tiles": {"tiles_per_head": m["tiles"],
                           "gflop": round(exec_flops / 1e9, 2),
                           "tflops_attention": round(exec_flops / (attn_ms * 1e-3) / 1e12, 2),
                           "note": "128 x 128 tiles with a visible key, each a dense QK^T and "
                                   "P.V on the tensor cores"},
        "tokens_per_s": round(world * S / (ms * 1e-3), 1),
        "kernel_ms": ({"mask_prepass_and_attn_kernel": round(attn_ms, 4),
                       "qk_prologue": round(kpro_ms + qpro_ms, 4)} if joint else
                      {"mask_prepass_and_attn_kernel": round(attn_ms, 4),
                       "k_prologue": round(kpro_ms, 4), "q_prologue": round(qpro_ms, 4)}),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4), "traffic": None,
                     "peak_kind": f"dense bf16 burst ({peak_src})",
                     "kernel": "ga_attn_masked_prepared (mask_prepass_kernel + "
                               "attn_kernel<mask>), algorithmic flops",
                     "algorithmic_flops": flops},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "schedule": "H2D, compute (ga_k_prologue + ga_attn_masked) and D2H on three "
                            "streams, device inputs and outputs double-buffered"},
        "gpu_launches": (3 if joint else 4) * args.steps, "clocks": clk,
        "device_status": status, "hidden_rows": hidden,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_masked(args.cpu_seconds, gpu_out=out)
    return line


def secondary_measurements(dev, rank, steps):
    """The two other long-context configurations, timed after the headline for a few steps
    each: the verify call (8 sequences x 16 rows over 65,536 cached keys, HBM-bound) and the
    sparse-selection masked call at S = 8192 (ga_attn_masked: mask prepass, query prologue,
    attention; keys prepared beforehand)."""
    from verify_gated_gqa_gb300 import binding as B
    if rank != 0:
        return None
    stream = torch.cuda.current_stream()
    peak_tf, peak_hbm, peak_src = measured_peaks()
    res = {}
    step, n_bytes = verify_setup(dev, SEED + 5, 8)
    ms = timed_steps(step, steps, 3, stream)
    gbs = n_bytes / (ms * 1e-3) / 1e9
    res["verify"] = {"workload": "ga_attn_verify, 8 sequences x 16 rows at positions "
                                 "65536..65551 over prepared K/V caches [65552, 2, 256] bf16",
                     "ms": round(ms, 4), "value": round(gbs, 1), "unit": "GB/s",
                     "algorithmic_bytes": n_bytes, "roofline_frac": round(gbs / peak_hbm, 4),
                     "peak": peak_hbm, "peak_kind": f"HBM copy ({peak_src})", "steps": steps}
    del step
    torch.cuda.empty_cache()
    m = masked_setup(dev, SEED + 7)
    out = torch.empty(S, HEADS * DIM, dtype=torch.bfloat16, device=dev)
    hid = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(B.ga_masked_workspace_bytes(S, S), dtype=torch.uint8, device=dev)

    def mstep():
        B.ga_attn_masked(m["qg"], m["k_prep"], m["v"], m["w_q"], m["cos"], m["sin"], m["mask"],
                         out=out, hidden_rows=hid, workspace=ws)

    ms = timed_steps(mstep, steps, 3, stream)
    tf = m["flops"] / (ms * 1e-3) / 1e12
    res["masked"] = {"workload": "ga_attn_masked at S=8192, stored mask: causal window of 128 "
                                 "keys plus 1024 random earlier keys per row",
                     "ms": round(ms, 4), "value": round(tf, 2), "unit": "TFLOP/s",
                     "algorithmic_gflop": round(m["flops"] / 1e9, 2),
                     "executed_tile_gflop": round(m["exec_flops"] / 1e9, 2),
                     "executed_tile_tflops": round(m["exec_flops"] / (ms * 1e-3) / 1e12, 2),
                     "roofline_frac": round(tf / peak_tf, 4), "peak": peak_tf,
                     "peak_kind": f"dense bf16 burst ({peak_src})", "steps": steps,
                     "device_status": B.ga_device_status()}
    return res


SEL_T, SEL_BUDGET, SEL_SETS = 8192, 2048, 4
# dram__bytes_read.sum + dram__bytes_write.sum of one select_mask_kernel launch at this
# size (ncu); L2 still holds most of the mask's writes when the launch ends
SELECT_TRAFFIC_BYTES = 48_163_840


def select_bytes(T=SEL_T, budget=SEL_BUDGET):
    """Algorithmic bytes of one selection-mask call over rows at positions 0 .. T-1: the
    candidate scores of every row that must select (more candidate blocks than it keeps;
    the others keep all of theirs and need no score), read once, and the T x T mask
    written once."""
    k = budget // 4
    read = sum(4 * (p // 4 + 1) for p in range(T) if p // 4 + 1 > k)
    return read + T * T


def run_select(args, world, rank, local):
    """The selection-mask producer: ga_select_mask over 8192 query rows and 8192 keys (2048
    blocks of 4 keys, N(0,1) fp32 scores), block_topk 512 (a budget of 2048 tokens). Each
    step takes the next of four input sets (scores 64 MiB + mask 64 MiB each), so the
    set a step touches has left L2 since its last use."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300 import synth
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    seed = SEED + 9 + rank
    k = SEL_BUDGET // 4
    scores = [synth.block_scores(seed + i, SEL_T, SEL_T // 4, device=dev) for i in range(SEL_SETS)]
    masks = [torch.empty(SEL_T, SEL_T, dtype=torch.uint8, device=dev) for _ in range(SEL_SETS)]
    n_bytes = select_bytes()
    it = [0]

    def step():
        i = it[0] % SEL_SETS
        it[0] += 1
        B.ga_select_mask(scores[i], SEL_T, k, mask=masks[i])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    if rank != 0:
        return None
    _, peak_hbm, peak_src = measured_peaks()
    gbs = n_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": "selection mask: HBM GB/s (8192 rows x 8192 keys, block_topk 512)",
        "value": round(world * gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) fp32 block scores)",
        "config": {"workload": "selection mask: scores [8192, 2048] fp32 -> mask [8192, 8192] "
                               "uint8, blocks of 4 keys, top 512 blocks per row AND causal",
                   "l2": f"{SEL_SETS} input sets of 128 MiB in rotation"},
        "rows_per_s": round(world * SEL_T / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                     "frac": round(gbs / peak_hbm, 4), "traffic": SELECT_TRAFFIC_BYTES,
                     "peak_kind": f"HBM copy ({peak_src})", "kernel": "select_mask_kernel",
                     "algorithmic_bytes": n_bytes},
        "gpu_launches": args.steps, "clocks": clk, "device_status": B.ga_device_status(),
    }


SMALL_CASES = [("S=64 causal", 64, True), ("S=2048 causal", 2048, True),
               ("S=2048 bidirectional", 2048, False)]


def run_small(args, world, rank, local):
    """The small prefill configurations: S = 64 causal (latency), S = 2048 causal and S = 2048
    bidirectional, each step the headline step's calls: both prologues (one ga_qk_prologue
    launch, or with --prologues side ga_k_prologue on a side stream beside ga_q_prologue,
    or serial), then ga_attn_prefill_prepared. Their inputs fit in L2, so every timed call
    follows a 256 MiB write that flushes it, and CUDA events bracket the step alone. The
    line's value is the S = 2048 causal TFLOP/s; `cases` holds all three, each with the
    attention call's own time beside the step's (also from a flushed L2)."""
    import statistics

    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300 import synth
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    cases = {}
    for name, n, causal in SMALL_CASES:
        qg, kraw, v, w_q, w_k = synth.attention_inputs(SEED + rank + n, n, n, device=dev)
        c, s_ = B.ga_rope_table_host(n)
        cos, sin = c.to(dev), s_.to(dev)
        k_prep = torch.empty_like(kraw)
        q_prep = torch.empty(n, HEADS, DIM, dtype=torch.bfloat16, device=dev)
        out = torch.empty(n, HEADS * DIM, dtype=torch.bfloat16, device=dev)
        side = torch.cuda.Stream(device=dev)

        def step():
            if args.prologues == "joint":
                B.ga_qk_prologue(kraw, w_k, qg, w_q, cos, sin, k_prep=k_prep, q_prep=q_prep)
            elif args.prologues == "serial":
                B.ga_k_prologue(kraw, w_k, cos, sin, k_prep=k_prep)
                B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)
            else:
                # the key prologue beside the query prologue; the attention waits for both
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    B.ga_k_prologue(kraw, w_k, cos, sin, k_prep=k_prep)
                B.ga_q_prologue(qg, w_q, cos, sin, q_prep=q_prep)
                stream.wait_stream(side)
            B.ga_attn_prefill_prepared(q_prep, qg, k_prep, v, 0, n, causal=causal, out=out)

        for _ in range(args.warmup):
            step()
        barrier(world)
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        # the same step captured once in a CUDA graph and replayed: the device's own time
        # without the host's per-call work
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        tg = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            tg.append(e0.elapsed_time(e1))
        # the attention call alone, its prepared inputs already written
        ta = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            B.ga_attn_prefill_prepared(q_prep, qg, k_prep, v, 0, n, causal=causal, out=out)
            e1.record(stream)
            torch.cuda.synchronize()
            ta.append(e0.elapsed_time(e1))
        barrier(world)
        ms = max_over_ranks(statistics.median(ts), world, dev)
        ms_g = max_over_ranks(statistics.median(tg), world, dev)
        ms_a = max_over_ranks(statistics.median(ta), world, dev)
        pairs = visible_pairs_causal(n, n) if causal else n * n
        flops = attention_flops(pairs)
        cases[name] = {"us_per_call": round(ms * 1e3, 2),
                       "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
                       "us_per_graph_replay": round(ms_g * 1e3, 2),
                       "tflops_graph": round(flops / (ms_g * 1e-3) / 1e12, 2),
                       "attn_us": round(ms_a * 1e3, 2),
                       "attn_tflops": round(flops / (ms_a * 1e-3) / 1e12, 2),
                       "algorithmic_gflop": round(flops / 1e9, 3)}
    clk = clocks.stop() if clocks else None
    if rank != 0:
        return None
    peak_tf, _, peak_src = measured_peaks()
    head = cases["S=2048 causal"]
    return {
        "metric": "causal prefill TFLOP/s at S=2048 (S=64 latency and S=2048 bidirectional in cases)",
        "value": round(world * head["tflops"], 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(head["us_per_call"] / 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": "small prefill configurations: S=64 causal, S=2048 causal, S=2048 "
                               "bidirectional; step = "
                               + {"joint": "ga_qk_prologue (both prologues, one launch)",
                                  "side": "ga_k_prologue (side stream) beside ga_q_prologue",
                                  "serial": "ga_k_prologue, ga_q_prologue"}[args.prologues]
                               + ", then ga_attn_prefill_prepared",
                   "l2": "flushed before every timed call (256 MiB write); median of the steps"},
        "cases": cases,
        "roofline": {"bound": "tensor", "achieved": head["tflops"], "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(head["tflops"] / peak_tf, 4),
                     "traffic": None, "peak_kind": f"dense bf16 burst ({peak_src})",
                     "kernel": "the S=2048 causal step (K prologue + Q prologue + attention)",
                     "algorithmic_flops": attention_flops(visible_pairs_causal(2048, 2048))},
        "gpu_launches": ((5 if args.prologues == "joint" else 7) * args.steps
                         * len(SMALL_CASES)), "clocks": clk,
        "device_status": B.ga_device_status(),
    }


def run_prefill_e4m3(args, world, rank, local):
    """Causal prefill at S = 8192 over e4m3 caches (prepared keys and values as e4m3 rows
    with an fp32 scale each, resident in HBM): the step is one ga_attn_prefill_e4m3 call,
    which widens both caches into its workspace, prepares the queries and attends."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    qg, kraw, v, w_q, w_k = make_inputs(dev, SEED + rank)
    c, s_ = B.ga_rope_table_host(S)
    cos, sin = c.to(dev), s_.to(dev)
    k_prep = B.ga_k_prologue(kraw, w_k, cos, sin)
    kq, ksc = B.ga_kv_quantize_e4m3(k_prep)
    vq, vsc = B.ga_kv_quantize_e4m3(v)
    del k_prep, kraw, v
    out = torch.empty(S, HEADS * DIM, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.ga_prefill_e4m3_workspace_bytes(S), dtype=torch.uint8, device=dev)

    def step():
        B.ga_attn_prefill_e4m3(qg, kq, ksc, vq, vsc, w_q, cos, sin, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    if rank != 0:
        return None
    peak_tf, _, peak_src = measured_peaks()
    tf = FLOPS_STEP / (ms * 1e-3) / 1e12
    return {
        "metric": "causal prefill over e4m3 K/V caches: TFLOP/s at S=8192",
        "value": round(world * tf, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": "causal gated GQA prefill, S=8192, over e4m3 caches of the "
                               "prepared keys and the values (fp32 scale per row); the call "
                               "widens them once into its workspace, then attends",
                   "l2": "inputs larger than L2 (qg 192 MiB read + out 96 MiB written per step)"},
        "tokens_per_s": round(world * S / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(tf / peak_tf, 4), "traffic": None,
                     "peak_kind": f"dense bf16 burst ({peak_src})",
                     "kernel": "ga_attn_prefill_e4m3 (2 widening launches + Q prologue + "
                               "attn_kernel), the whole call",
                     "algorithmic_flops": FLOPS_STEP},
        "gpu_launches": 4 * args.steps, "clocks": clk, "device_status": B.ga_device_status(),
    }


B_LENS = [512 * (1 + b % 8) for b in range(16)]   # 16 prompts of 512 .. 4096 tokens
B_PAGE = 256


def run_batch(args, world, rank, local):
    """Batched causal prefill: 16 prompts of 512 to 4096 tokens (36,864 rows in all) in one
    ga_attn_prefill_batch call over prepared caches in 256-position pages scattered over two
    page pools (seeded random order); the step is the call (query prologue + attention)."""
    from verify_gated_gqa_gb300 import binding as B
    from verify_gated_gqa_gb300 import synth
    from verify_gated_gqa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    seed = SEED + 7 + rank
    tmax = max(B_LENS)
    c, s = B.ga_rope_table_host(tmax)
    cos, sin = c.to(dev), s.to(dev)
    w_q = synth.normal_bf16(seed, "w_q", (DIM,), sigma=0.1, device=dev)
    w_k = synth.normal_bf16(seed, "w_k", (DIM,), sigma=0.1, device=dev)
    need = [-(-L // B_PAGE) for L in B_LENS]
    order = torch.randperm(sum(need), generator=torch.Generator().manual_seed(seed))
    k_pool = torch.zeros(sum(need), B_PAGE, KV_HEADS, DIM, dtype=torch.bfloat16, device=dev)
    v_pool = torch.zeros_like(k_pool)
    table = torch.full((len(B_LENS), max(need)), -1, dtype=torch.int32)
    i = 0
    seqs = []   # the same prompts as contiguous caches, for one-call-per-prompt timing
    for b, L in enumerate(B_LENS):
        k_raw = synth.normal_bf16(seed, "k", (L, KV_HEADS, DIM), sub=b, device=dev)
        k_prep = torch.empty_like(k_raw)
        B.ga_k_prologue(k_raw, w_k, cos, sin, k_prep=k_prep)
        v = synth.normal_bf16(seed, "v", (L, KV_HEADS, DIM), sub=b, device=dev)
        seqs.append((k_prep, v))
        for p in range(need[b]):
            pg = int(order[i])
            i += 1
            table[b, p] = pg
            lo, hi = p * B_PAGE, min((p + 1) * B_PAGE, L)
            k_pool[pg, :hi - lo] = k_prep[lo:hi]
            v_pool[pg, :hi - lo] = v[lo:hi]
    table = table.to(dev)
    qg = torch.cat([synth.normal_bf16(seed, "qg", (L, HEADS, 2 * DIM), sub=b, device=dev)
                    for b, L in enumerate(B_LENS)])
    starts = [0]
    for L in B_LENS:
        starts.append(starts[-1] + L)
    out = torch.empty(qg.shape[0], HEADS * DIM, dtype=torch.bfloat16, device=dev)
    flops = sum(attention_flops(visible_pairs_causal(L, L)) for L in B_LENS)

    def step():
        B.ga_attn_prefill_batch(qg, starts, [0] * len(B_LENS), k_pool, v_pool, table, w_q, cos,
                                sin, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps

    # context: the same prompts as one ga_attn_prefill call each (not the metric)
    def separate():
        for b, L in enumerate(B_LENS):
            B.ga_attn_prefill(qg[starts[b]:starts[b + 1]], seqs[b][0], seqs[b][1], w_q, cos, sin,
                              0, L, out=out[starts[b]:starts[b + 1]])

    for _ in range(3):
        separate()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_sep = max(3, min(args.steps, 20))
    e0.record(stream)
    for _ in range(n_sep):
        separate()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_sep = e0.elapsed_time(e1) / n_sep
    if rank != 0:
        return None
    peak_bf16, _, peak_src = measured_peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    return {
        "metric": "batched causal prefill attention TFLOP/s (16 prompts of 512..4096 tokens)",
        "value": round(world * tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": f"batched causal gated GQA prefill: {len(B_LENS)} prompts of "
                               f"{min(B_LENS)}..{max(B_LENS)} tokens ({starts[-1]} rows), 24q/2kv "
                               f"heads, d=256, caches in pages of {B_PAGE} positions scattered "
                               "over two page pools",
                   "l2": f"inputs larger than L2 (qg {qg.numel() * 2 / 2**20:.0f} MiB)"},
        "tokens_per_s": round(world * starts[-1] / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak_bf16,
                     "unit": "TFLOP/s", "frac": round(tflops / peak_bf16, 4), "traffic": None,
                     "peak_kind": f"dense bf16 burst ({peak_src})",
                     "kernel": "ga_attn_prefill_batch (query prologue + attn_kernel<batch>)",
                     "algorithmic_flops": flops},
        "gpu_launches": 2 * args.steps, "clocks": clk, "device_status": B.ga_device_status(),
        "one_call_per_prompt": {"ms": round(ms_sep, 4), "calls": len(B_LENS),
                                "note": "the same prompts as contiguous caches, one "
                                        "ga_attn_prefill each; context, not the metric"},
    }


# Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu captures
# summarised in profiles/attn_kernel_causal_s8192.md (218,658,048 + 62,062,080, the causal
# variant as CTA pairs) and profiles/attn_kernel_verify_8x16_l65536.md (1,075,831,040 +
# 7,228,672, the verify variant of attn_kernel); each is to be set to None whenever its
# kernel changes until it is captured again.
ATTN_TRAFFIC_BYTES = 280_720_128
VERIFY_ATTN_TRAFFIC_BYTES = 1_083_059_712


# ---------------------------------------------------------------- the oracle as baseline
def oracle_sample_step(qg, kraw, v, w_q, w_k, cos, sin, rows):
    """One bounded sample of the workload in the CPU oracle: the K prologue over all keys
    and the causal attention of the listed query rows (all 24 heads)."""
    from oracle import ga_oracle as O
    kp = O.prep_keys(kraw, w_k, cos, sin)
    return O.prefill(qg, kp, v, w_q, cos, sin, 0, S, True, "R1", rows=rows)


def _oracle_inputs():
    import numpy as np  # noqa: F401
    from oracle import ga_oracle as O
    from verify_gated_gqa_gb300 import synth
    qg, k, v, w_q, w_k = synth.attention_inputs(SEED, S, S)
    f = lambda t: t.double().numpy()
    cos, sin = O.rope_tables(S)
    return f(qg), f(k), f(v), f(w_q), f(w_k), cos, sin


def _threads_used():
    try:
        from threadpoolctl import threadpool_info
        n = max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


class _ParityTally:
    """Parity of the GPU output on the oracle's sampled rows (the tests' element-wise check:
    2 bf16 ulp + 1e-5, with its ambiguous-rounding rule), summed over the samples."""

    def __init__(self):
        self.n = self.bad = self.pairs = self.off = self.explained = 0
        self.over = 0.0
        self.max_ulp = 0.0
        self.passed = True

    def add(self, ref, got):
        import contextlib
        import io
        with contextlib.redirect_stdout(io.StringIO()):
            try:
                st = ref.check(got)
            except AssertionError:
                self.passed = False
                return
        self.n += st["n"]
        self.bad += st["bad"]
        self.over += st["over_1ulp"] * st["n"]
        self.max_ulp = max(self.max_ulp, st["max_ulp"])
        self.pairs += len(ref.rows) * len(ref.heads)
        self.off += st["rows_off_oracle"]
        self.explained += st["explained_by_ambiguous_rounding"]

    def summary(self, what):
        return {"what": what, "elements": self.n, "bad": self.bad,
                "over_1ulp": round(self.over / max(self.n, 1), 6),
                "max_ulp": round(self.max_ulp, 2), "pairs": self.pairs,
                "pairs_off_oracle": self.off, "explained_by_ambiguous_rounding": self.explained,
                "passed": self.passed,
                "tolerance": "|gpu - oracle| <= 2 bf16 ulp(oracle) + 1e-5 per element"}


def cpu_baseline(seconds: float, gpu_out=None):
    """The oracle on a bounded sample of the headline workload (random query rows, all 24
    heads, with the K prologue over all keys), timed on the host cores. When the GPU output
    of the same inputs is given, each sampled row is also checked against it (untimed)."""
    import numpy as np
    from oracle import ga_oracle as O
    from tests.parity import AttnRef
    qg, kraw, v, w_q, w_k, cos, sin = _oracle_inputs()
    rng = np.random.default_rng(0)
    pairs = 0
    spent = 0.0
    n_rows = 0
    tally = _ParityTally()
    got = gpu_out.cpu() if gpu_out is not None else None
    while spent < seconds:
        rows = np.sort(rng.choice(S, 16, replace=False))
        t0 = time.perf_counter()
        kp = O.prep_keys(kraw, w_k, cos, sin)
        ref = AttnRef(qg, kp, v, w_q, cos, sin, 0, S, "causal", rows=rows)
        spent += time.perf_counter() - t0
        if got is not None:
            tally.add(ref, got[torch.as_tensor(rows)])
        pairs += int((rows + 1).sum())
        n_rows += 16
    res = {"value": round(attention_flops(pairs) / spent / 1e12, 6), "unit": UNIT,
           "cores": _threads_used(), "kind": "oracle",
           "sample": f"{n_rows} random query rows x 24 heads of the S=8192 causal pass, each "
                     f"16-row batch with the K prologue over all 8192 keys; {spent:.1f} s"}
    if got is not None:
        res["parity"] = tally.summary("the timed launch's output on the sampled rows")
    return res


def cpu_baseline_masked(seconds: float, gpu_out=None):
    """The oracle on the masked workload: the key prologue over all 8192 keys and the
    stored-mask attention of 16 random query rows (all 24 heads) per batch; with the GPU
    output given, each sampled row is also checked against it (untimed)."""
    import numpy as np
    from oracle import ga_oracle as O
    from tests.parity import AttnRef
    from verify_gated_gqa_gb300 import synth
    qg, k, v, w_q, w_k = synth.attention_inputs(SEED + 7, S, S)
    mask = synth.selection_mask(SEED + 7, S, window=M_WINDOW, n_random=M_RANDOM).numpy()
    f = lambda t: t.double().numpy()
    qg, k, v, w_q, w_k = f(qg), f(k), f(v), f(w_q), f(w_k)
    cos, sin = O.rope_tables(S)
    rng = np.random.default_rng(0)
    pairs = n_rows = 0
    spent = 0.0
    tally = _ParityTally()
    got = gpu_out.cpu() if gpu_out is not None else None
    while spent < seconds:
        rows = np.sort(rng.choice(S, 16, replace=False))
        t0 = time.perf_counter()
        kp = O.prep_keys(k, w_k, cos, sin)
        ref = AttnRef(qg, kp, v, w_q, cos, sin, 0, S, "mask", mask=mask, rows=rows)
        spent += time.perf_counter() - t0
        if got is not None:
            tally.add(ref, got[torch.as_tensor(rows)])
        pairs += int((mask[rows] != 0).sum())
        n_rows += 16
    res = {"value": round(attention_flops(pairs) / spent / 1e12, 6), "unit": UNIT,
           "cores": _threads_used(), "kind": "oracle",
           "sample": f"{n_rows} random query rows x 24 heads of the S=8192 masked pass, each "
                     f"16-row batch with the K prologue over all 8192 keys; {spent:.1f} s"}
    if got is not None:
        res["parity"] = tally.summary("the timed launch's output on the sampled rows")
    return res


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this machine's host cores."""
    if rank != 0:
        return None
    import numpy as np
    data = _oracle_inputs()
    rng = np.random.default_rng(1)
    per_step_rows = 2

    def one():
        rows = np.sort(rng.choice(S, per_step_rows, replace=False))
        oracle_sample_step(*data, rows)
        return int((rows + 1).sum())

    for _ in range(args.warmup):
        one()
    pairs = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        pairs += one()
    dt = time.perf_counter() - t0
    value = attention_flops(pairs) / dt / 1e12
    sample = (f"{per_step_rows} random query rows x 24 heads of the S=8192 causal pass per "
              f"step, with the K prologue over all 8192 keys")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.1) norm weights)",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": S,
                   "parallelism": "none (CPU oracle)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _threads_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default="prefill",
                    choices=["prefill", "verify", "verify_paged", "verify_e4m3", "batch",
                             "select", "prefill_e4m3", "small", "masked"],
                    help="prefill: the headline S=8192 causal step; verify: 8 x 16 rows over "
                         "65,536 cached keys; verify_paged: the same over paged caches; "
                         "verify_e4m3: the same over e4m3 caches; batch: 16 prompts of "
                         "512..4096 tokens in one batched call; select: the selection-mask "
                         "producer at 8192 x 8192, block_topk 512; prefill_e4m3: the "
                         "headline causal step over e4m3 caches; small: S=64 and S=2048 "
                         "(causal and bidirectional) with L2 flushed before each call; masked: "
                         "sparse-selection masked attention at S=8192 (window 128 + 1024 "
                         "random keys per row)")
    ap.add_argument("--verify-seqs", type=int, default=8)
    ap.add_argument("--no-secondary", action="store_true",
                    help="prefill: skip the verify and masked measurements after the headline "
                         "(for profiling runs)")
    ap.add_argument("--prologues", choices=("joint", "side", "serial"), default="joint",
                    help="prefill and small: both prologues in one launch (joint), the key "
                         "prologue on a side stream beside the query prologue (side), or "
                         "one after the other (serial)")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.workload in ("verify", "verify_paged", "verify_e4m3"):
        line = run_verify(args, world, rank, local)
    elif args.workload == "batch":
        line = run_batch(args, world, rank, local)
    elif args.workload == "select":
        line = run_select(args, world, rank, local)
    elif args.workload == "prefill_e4m3":
        line = run_prefill_e4m3(args, world, rank, local)
    elif args.workload == "small":
        line = run_small(args, world, rank, local)
    elif args.workload == "masked":
        line = run_masked(args, world, rank, local)
    else:
        line = run_gpu(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
