#!/usr/bin/env python3
"""Benchmark: one step = routing layout + dispatch copy epilogue + combine.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
    python bench.py --impl reference ...     (the CPU oracle, timed on host cores)

Prints ONE JSON line (rank 0).  The workload is the 4096-token, hidden-7168
prefill batch (group-limited top-8 routing over 256 experts in 8 logical
ranks; FP8 dispatch with column-major scales into the expanded layout,
alignment 128, zero padding, exact allocation; BF16 combine).  ``value`` is
algorithmic HBM GB/s of the whole step (layout + dispatch + combine bytes
over their device time, L2 flushed before every stage); ``e2e`` is the same
metric through the C ABI with the step's inputs copied in from pinned host
memory and the combined output copied back, inside the timed region.

Multi-GPU: every rank runs an independent replica (the single-GPU path does
not shard: logical ranks live in one HBM), times are the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ep_workloads as W  # noqa: E402

METRIC = "dispatch & combine HBM GB/s (% of GB300 peak) and tokens/s, 1 GPU"
L2_FLUSH_BYTES = 256 << 20
REFERENCE_BUDGET_S = 120.0   # CPU time of a whole `--impl reference` run


# ---------------------------------------------------------------------------
# Algorithmic bytes (what each stage must move; never the allocation size)
# ---------------------------------------------------------------------------
def stage_bytes(wl: W.Workload, T: int, topk_idx, rows_valid: int, rows_padding: int,
                rows_distinct_read: int, with_recv_w=True, with_recv_idx=True,
                combine_weights=True, bias_rows=0, expert_bias=False) -> dict:
    """Bytes per stage for one batch.

    layout   : topk_idx read (8 B/slot), dst written (4 B/slot), int32 copy of
               topk_idx (4 B/slot), source metadata (8 B/row), is_token_in_rank
               (1 B per token and rank).
    dispatch : each active source row read once (2H), per slot dst + idx +
               weight reads (12 B), per destination row its payload (H or 2H),
               scales (4 B per 128 elements, FP8), weight(s) and local expert
               ids; padding rows their zero payload, scales and weight.
    combine  : each distinct expert-output row read once (2H), per slot dst
               and weight reads (8 B), output write (2H per token), biases.
    """
    K, H, R = wl.num_topk, wl.hidden, wl.num_ranks
    idx = topk_idx
    valid = idx >= 0
    t_active = int(valid.any(dim=1).sum())
    b = 1 if wl.use_fp8 else 2
    sf = 4 * (H // 128) if wl.use_fp8 else 0
    rows = rows_valid
    w_row = (4 if wl.do_expand else 4 * K) if with_recv_w else 0
    i_row = (0 if wl.do_expand else 4 * K) if with_recv_idx else 0
    layout = T * K * (8 + 4 + 4) + rows * 8 + T * R
    dispatch = (t_active * H * 2 + T * K * 12 + rows * (H * b + sf + w_row + i_row)
                + rows_padding * ((H * b + sf if wl.do_zero_padding else 0) + (4 if with_recv_w else 0)))
    combine = (rows_distinct_read * H * 2 + T * K * (8 if combine_weights else 4) + T * H * 2
               + bias_rows * H * 2 + (wl.num_experts * H * 2 if expert_bias else 0))
    return {"layout": layout, "dispatch": dispatch, "combine": combine}


def backward_bytes(wl: W.Workload, T: int, topk_idx, rows_valid: int, rows_padding: int,
                   rows_distinct_read: int) -> dict:
    """Bytes of the backward pair for one batch.

    combine_backward  : BF16 dispatch of the gradient without weights: each
                        active source row read once (2H), per slot dst + idx
                        reads (8 B), each destination row written (2H), padding
                        rows zeroed (2H, with zero padding).
    dispatch_backward : unweighted combine (each distinct row read once, 2H;
                        dst 4 B/slot; output 2H per token) plus the weight
                        reduction (dst 4 B/slot, the row's weight gradient,
                        4 B expanded or 4K B rank layout, result 4 B/slot).
    """
    K, H = wl.num_topk, wl.hidden
    t_active = int((topk_idx >= 0).any(dim=1).sum())
    comb_b = (t_active * H * 2 + T * K * 8 + rows_valid * H * 2
              + (rows_padding * H * 2 if wl.do_expand and wl.do_zero_padding else 0))
    g_row = 4 if wl.do_expand else 4 * K
    disp_b = (rows_distinct_read * H * 2 + T * K * 4 + T * H * 2
              + T * K * 8 + rows_valid * g_row)
    return {"combine_backward": comb_b, "dispatch_backward": disp_b}


def prequantised_bytes(wl: W.Workload, T: int, topk_idx, rows_valid: int,
                       rows_padding: int) -> int:
    """Bytes of dispatch with a pre-quantised FP8 input: each active token's
    e4m3 row (H) and scales (4 B per 128 elements) read once, 12 B per slot,
    per destination row its payload and scales plus weight(s) and local
    expert ids, per padding row its zero payload, scales and weight."""
    K, H = wl.num_topk, wl.hidden
    t_active = int((topk_idx >= 0).any(dim=1).sum())
    sf = 4 * (H // 128)
    w_row = 4 if wl.do_expand else 4 * K
    i_row = 0 if wl.do_expand else 4 * K
    return (t_active * (H + sf) + T * K * 12 + rows_valid * (H + sf + w_row + i_row)
            + rows_padding * ((H + sf if wl.do_zero_padding else 0) + 4))


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# Distributed helpers (replicas only; no collective on the data path)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, ws: int, device="cpu") -> float:
    if ws <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, ws: int, device="cpu") -> float:
    if ws <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "combine_topk_idx_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            s = line.split("#")[0].split()
            if len(s) >= 4 and s[0] == kernel and s[1] == workload:
                src = {"dispatch": "ep_dispatch.cu", "combine": "ep_combine.cu",
                       "layout": "ep_layout.cu"}[kernel]
                if s[3] != kernel_source_hash(src):
                    return None
                return int(s[2])
    return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_layout(wl: W.Workload, idx, M: int):
    from oracle import ep_oracle as O
    if wl.fixed_capacity:
        return O.layout_fixed_capacity(idx, wl.num_experts, wl.num_ranks, M)
    return O.layout(idx, wl.num_experts, wl.num_ranks, M, wl.expert_alignment, wl.do_expand, True)


def sample_tokens_per_rank(wl: W.Workload, T: int) -> int:
    """M for a CPU sample of T tokens: the workload's, except that a
    fixed-capacity sample uses the smallest capacity that holds it (the
    oracle materialises every row of every expert's slab)."""
    if wl.fixed_capacity:
        return max(1, -(-T // wl.num_ranks))
    return wl.num_max_tokens_per_rank


def oracle_step(wl: W.Workload, inp: dict, y_bits):
    from oracle import ep_oracle as O
    idx = inp["topk_idx"].numpy()
    lay = oracle_layout(wl, idx, sample_tokens_per_rank(wl, idx.shape[0]))
    xb = inp["x"].view(torch.int16).numpy().view("uint16")
    eb = inp["expert_bias"]
    eb = None if eb is None else eb.view(torch.int16).numpy().view("uint16")
    O.dispatch(lay, xb, inp["topk_weights"].numpy(), wl.use_fp8, wl.col_major_sf,
               wl.do_zero_padding)
    O.combine(lay, y_bits, inp["topk_weights"].numpy(), None, None, eb)
    return lay


def oracle_setup(wl: W.Workload, sample_tokens: int, seed: int = 0):
    """Inputs of a CPU sample: the first ``sample_tokens`` tokens, and expert
    outputs for just the rows their routing references."""
    import numpy as np
    T = min(sample_tokens, wl.num_tokens)
    inp = W.make_inputs(wl, seed=seed, num_tokens=T)
    lay0 = oracle_layout(wl, inp["topk_idx"].numpy(), sample_tokens_per_rank(wl, T))
    dst = lay0["dst_buffer_slot_idx"]
    need = np.unique(dst[dst >= 0])
    y_bits = np.zeros((max(lay0["rows_alloc"], 1), wl.hidden), dtype=np.uint16)
    if need.size:
        y_bits[need] = W.hashed_bf16_rows(torch.from_numpy(need), wl.hidden, 7).view(
            torch.int16).numpy().view(np.uint16)
    return T, inp, y_bits


def oracle_sample_text(wl: W.Workload, T: int, seed: int, n: int) -> str:
    return (f"first {T} tokens of the {wl.name} workload (seed {seed}), full step "
            f"(layout + dispatch + combine) on 1 core, {n} pass(es)"
            + (f"; expert capacity {sample_tokens_per_rank(wl, T) * wl.num_ranks} "
               f"rows (the smallest that holds the sample)" if wl.fixed_capacity else ""))


def time_oracle(wl: W.Workload, sample_tokens: int, budget_s: float, seed: int = 0):
    """Run the oracle, as it stands, on the first ``sample_tokens`` tokens of
    the workload until ``budget_s`` seconds pass (at least once)."""
    T, inp, y_bits = oracle_setup(wl, sample_tokens, seed)
    n, t0 = 0, time.perf_counter()
    lay = None
    while True:
        lay = oracle_step(wl, inp, y_bits)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = (time.perf_counter() - t0) / n
    by = bytes_from_layout(wl, T, inp["topk_idx"], lay)
    total = sum(by.values())
    return {"gbs": total / el / 1e9, "tokens_per_s": T / el, "sec_per_step": el, "steps": n,
            "sample": oracle_sample_text(wl, T, seed, n)}


def _oracle_worker(job):
    """One process of the all-cores oracle timing (spawned, one thread)."""
    name, tokens, budget, seed = job
    torch.set_num_threads(1)
    r = time_oracle(W.WORKLOADS[name], tokens, budget, seed=seed)
    return r["gbs"], r["tokens_per_s"]


def time_oracle_all_cores(wl: W.Workload, sample_tokens: int, budget_s: float, seed: int):
    """The oracle on every host core at once: one spawned process per core,
    each timing its own sample (seeds seed, seed + 1, ...); the aggregate
    throughput is the sum.  None if no process pool can be started."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_worker, [(wl.name, sample_tokens, budget_s, seed + i)
                                             for i in range(n)])
    except Exception:
        return None
    return {"value": round(sum(g for g, _ in res), 4), "unit": "GB/s", "cores": n,
            "kind": "oracle", "tokens_per_s": round(sum(t for _, t in res), 1),
            "cpu_model": cpu_model(),
            "sample": f"{n} processes, each the first {min(sample_tokens, wl.num_tokens)} tokens "
                      f"of the {wl.name} workload with its own seed, for {budget_s:g} s"}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def bytes_from_layout(wl, T, topk_idx, lay: dict) -> dict:
    import numpy as np
    dst = lay["dst_buffer_slot_idx"]
    rows_valid = int(lay["num_expanded_tokens"] - (lay["cnt_expert_aligned"] - lay["cnt_expert"]).sum()) \
        if wl.do_expand else int(lay["num_recv_tokens"])
    rows_pad = int((lay["cnt_expert_aligned"] - lay["cnt_expert"]).sum()) if wl.do_expand else 0
    distinct = int(np.unique(dst[dst >= 0]).size)
    return stage_bytes(wl, T, topk_idx, rows_valid, rows_pad, distinct,
                       expert_bias=wl.expert_bias_std > 0)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, ws, rank, local):
    import numpy as np
    import combine_topk_idx_gb300 as ep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    ep.load_library()
    wl = W.WORKLOADS[args.workload]
    T, H = wl.num_tokens, wl.hidden
    inp = W.make_inputs(wl, seed=args.seed)
    idx_h, w_h, x_h = inp["topk_idx"], inp["topk_weights"], inp["x"]
    idx, w, x = idx_h.to(dev), w_h.to(dev), x_h.to(dev)
    eb = inp["expert_bias"].to(dev) if inp["expert_bias"] is not None else None
    cfg = ep.make_config(T, wl.num_topk, wl.num_experts, wl.num_ranks, H,
                         wl.num_max_tokens_per_rank, wl.expert_alignment, wl.do_expand,
                         wl.do_zero_padding, wl.do_cpu_sync, wl.use_fp8, wl.col_major_sf,
                         fixed_capacity=wl.fixed_capacity)
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one, so that the
        # next timed stage starts with a cold L2 holding no dirty lines
        flush_w.zero_()
        flush_r.sum()

    # Expert outputs for combine (identity experts): y = dequantised / copied
    # recv_x, produced once, untimed, by torch ops (not part of the path).
    h0 = ep.ep_layout(cfg, idx)
    out0 = ep.alloc_recv(h0, with_weights=True, with_idx=True, zero=True)
    ep.ep_dispatch(h0, x, w, **out0)
    rows = h0.rows_alloc
    if wl.use_fp8:
        q = out0["recv_x"].view(torch.float8_e4m3fn).float()
        nb = H // 128
        sf = out0["recv_sf"]
        if wl.col_major_sf:
            s = sf.view(nb, -1)[:, :rows].t()
        else:
            s = sf.view(rows, nb)
        y = (q.view(rows, nb, 128) * s.unsqueeze(-1)).view(rows, H).to(torch.bfloat16)
        del q
    else:
        y = out0["recv_x"].clone()
    g0 = {n: h0.tensor(n).cpu() for n in ("dst_buffer_slot_idx", "cnt_expert",
                                            "cnt_expert_aligned", "totals")}
    torch.cuda.synchronize()
    dst = g0["dst_buffer_slot_idx"]
    pad_rows = int((g0["cnt_expert_aligned"] - g0["cnt_expert"]).sum()) if wl.do_expand else 0
    total_rows = int(g0["totals"][1] if wl.do_expand else g0["totals"][0])
    valid_rows = total_rows - pad_rows
    distinct = int(torch.unique(dst[dst >= 0]).numel())
    by = stage_bytes(wl, T, idx_h, valid_rows, pad_rows, distinct,
                     expert_bias=eb is not None)
    out_comb = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    grad_recv_w = out0["recv_topk_weights"].clone()
    h0.free()
    del out0

    def one_step(timed: bool, ev=None, flush=True):
        if flush:
            flush_l2()
        if timed:
            ev[0].record(stream)
        h = ep.ep_layout(cfg, idx)
        if timed:
            ev[1].record(stream)
        out = ep.alloc_recv(h, with_weights=True, with_idx=True)
        if flush:
            flush_l2()
        if timed:
            ev[2].record(stream)
        ep.ep_dispatch(h, x, w, **out)
        if timed:
            ev[3].record(stream)
        if flush:
            flush_l2()
        if timed:
            ev[4].record(stream)
        ep.ep_combine(h, y, w, None, None, eb, out=out_comb)
        if timed:
            ev[5].record(stream)
        h.free()
        return h.rows_alloc

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    barrier(ws)
    torch.cuda.synchronize()
    launches = 0
    for i in range(args.steps):
        r = one_step(True, evs[i])
        # layout: count + assign; dispatch: the copy kernel (+ the column-major
        # scale gather for FP8); combine: one kernel
        launches += 2 + ((1 + int(wl.use_fp8 and wl.col_major_sf)) if r > 0 else 0) + \
            (1 if T > 0 else 0)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    lay_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dis_ms = [e[2].elapsed_time(e[3]) for e in evs]
    com_ms = [e[4].elapsed_time(e[5]) for e in evs]
    step_ms = statistics.mean(a + b + c for a, b, c in zip(lay_ms, dis_ms, com_ms))
    step_ms_max = max_over_ranks(step_ms, ws, dev)
    total_bytes = sum(by.values())
    value = total_bytes * ws / (step_ms_max * 1e-3) / 1e9

    # Secondary: warm L2 (no flush between stages), same step, untimed warm-up.
    warm_steps = max(8, args.steps // 8)
    for _ in range(3):
        one_step(False, flush=False)
    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(warm_steps)]
    torch.cuda.synchronize()
    for i in range(warm_steps):
        one_step(True, wev[i], flush=False)
    torch.cuda.synchronize()
    warm = {k: statistics.mean(e[a].elapsed_time(e[b]) for e in wev)
            for k, a, b in (("layout", 0, 1), ("dispatch", 2, 3), ("combine", 4, 5))}
    # Host wall time of the layout call on an idle GPU (with do_cpu_sync it
    # includes the count wait).
    layout_host_s = []
    for _ in range(20):
        torch.cuda.synchronize()
        t_host = time.perf_counter()
        h = ep.ep_layout(cfg, idx)
        layout_host_s.append(time.perf_counter() - t_host)
        h.free()
    torch.cuda.synchronize()

    # e2e through the C ABI with host buffers: every step copies its inputs
    # (topk_idx, topk_weights, x) in from pinned host memory and its combined
    # output back out.  Steps rotate over three streams and buffer sets, and
    # the next step's input copies are enqueued before this step's layout
    # (whose count wait blocks the host), so one step's copies overlap the
    # neighbouring steps' kernels and copies, as a serving loop would run them.
    idx_pin, w_pin, x_pin = idx_h.pin_memory(), w_h.pin_memory(), x_h.pin_memory()
    nbuf = 3
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(nbuf)]
    e2e_bufs = [{"idx": torch.empty_like(idx), "w": torch.empty_like(w), "x": torch.empty_like(x),
                 "out": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                 "out_pin": torch.empty((T, H), dtype=torch.bfloat16).pin_memory()}
                for _ in range(nbuf)]

    def e2e_copy_in(i):
        b = e2e_bufs[i % nbuf]
        with torch.cuda.stream(e2e_streams[i % nbuf]):
            b["idx"].copy_(idx_pin, non_blocking=True)
            b["w"].copy_(w_pin, non_blocking=True)
            b["x"].copy_(x_pin, non_blocking=True)

    def e2e_step(i):
        st = e2e_streams[i % nbuf]
        b = e2e_bufs[i % nbuf]
        with torch.cuda.stream(st):
            h = ep.ep_layout(cfg, b["idx"], stream=st)
            out = ep.alloc_recv(h, with_weights=True, with_idx=True)
            ep.ep_dispatch(h, b["x"], b["w"], **out, stream=st)
            ep.ep_combine(h, y, b["w"], None, None, eb, out=b["out"], stream=st)
            b["out_pin"].copy_(b["out"], non_blocking=True)
            h.free()

    def e2e_run(n):
        for st in e2e_streams:
            st.wait_stream(stream)
        e2e_copy_in(0)
        for i in range(n):
            if i + 1 < n:
                e2e_copy_in(i + 1)
            e2e_step(i)
        for st in e2e_streams:
            stream.wait_stream(st)

    e2e_run(max(4, args.warmup))
    torch.cuda.synchronize()
    e2e_steps = max(8, args.steps // 4)
    barrier(ws)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_l2()
    e_s.record(stream)
    e2e_run(e2e_steps)
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, ws, dev)
    barrier(ws)

    # Backward pair on one handle (layout untimed): combine_backward dispatches
    # a [T, H] gradient, dispatch_backward combines a [rows, H] gradient and
    # reduces the weight gradients.  L2 is flushed before each timed call.
    bwd_by = backward_bytes(wl, T, idx_h, valid_rows, pad_rows, distinct)
    hb = ep.ep_layout(cfg, idx)
    g_recv = torch.empty((hb.rows_alloc, H), dtype=torch.bfloat16, device=dev)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    g_w = torch.empty((T, wl.num_topk), dtype=torch.float32, device=dev)

    def bwd_step(ev=None):
        flush_l2()
        if ev:
            ev[0].record(stream)
        ep.ep_combine_backward(hb, x, g_recv)
        if ev:
            ev[1].record(stream)
        flush_l2()
        if ev:
            ev[2].record(stream)
        ep.ep_dispatch_backward(hb, y, grad_recv_w, g_x, g_w)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        bwd_step()
    bwd_steps = max(8, args.steps // 4)
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(bwd_steps)]
    torch.cuda.synchronize()
    for i in range(bwd_steps):
        bwd_step(bev[i])
    torch.cuda.synchronize()
    cb_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in bev)
    db_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in bev)
    del g_recv, g_x, g_w

    # Dispatch of a pre-quantised input (FP8 workloads): x as e4m3 bytes with
    # column-major TMA-aligned fp32 scales, made once by torch, untimed.
    pq = None
    if wl.use_fp8:
        nb = H // 128
        xb = x.float().view(T, nb, 128)
        sc = xb.abs().amax(-1) / 448.0
        sc = torch.where(sc > 0, sc, torch.ones_like(sc))
        xq = (xb / sc.unsqueeze(-1)).to(torch.float8_e4m3fn).view(T, H)
        st = -(-max(T, 1) // 4) * 4
        sf_store = torch.zeros((nb, st), dtype=torch.float32, device=dev)
        sf_store[:, :T] = sc.t()
        xs = sf_store[:, :T].t()
        del xb
        pq_out = ep.alloc_recv(hb, with_weights=True, with_idx=True)
        pq_by = prequantised_bytes(wl, T, idx_h, valid_rows, pad_rows)

        def pq_step(ev=None):
            flush_l2()
            if ev:
                ev[0].record(stream)
            ep.ep_dispatch_fp8(hb, xq, xs, w, **pq_out)
            if ev:
                ev[1].record(stream)

        for _ in range(args.warmup):
            pq_step()
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(bwd_steps)]
        torch.cuda.synchronize()
        for i in range(bwd_steps):
            pq_step(pev[i])
        torch.cuda.synchronize()
        pq_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in pev)
        pq = {"steps": bwd_steps, "ms": round(pq_ms, 5), "bytes": pq_by,
              "gbs": round(pq_by / pq_ms / 1e6, 1),
              "input_sf": "column-major TMA-aligned",
              "gpu_launches": bwd_steps * (1 + int(wl.col_major_sf))}
        del pq_out, xq, sf_store
    hb.free()

    peaks = load_peaks()
    d_ms, c_ms = statistics.mean(dis_ms), statistics.mean(com_ms)
    dom = "combine" if c_ms >= d_ms else "dispatch"
    dom_ms = c_ms if dom == "combine" else d_ms
    achieved = by[dom] / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(dom, wl.name)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32", "data": "synthetic (seeded generators; no dataset on the pages)",
        "config": {"workload": wl.name, "tokens": T, "hidden": H, "experts": wl.num_experts,
                   "logical_ranks": wl.num_ranks, "topk": wl.num_topk,
                   "expert_alignment": wl.expert_alignment, "do_expand": wl.do_expand,
                   "fp8_dispatch": wl.use_fp8, "col_major_sf": wl.col_major_sf,
                   "do_cpu_sync": wl.do_cpu_sync, "routing": wl.routing,
                   "l2": "flushed before each stage (256 MiB write, then 256 MiB read); "
                         "times are device events",
                   "parallelism": f"replicas x{ws}"},
        "tokens_per_s": round(T * ws / (step_ms_max * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * value / ws / peaks["hbm_gbs"], 2),
        "stages": {
            "layout": {"ms": round(statistics.mean(lay_ms), 5), "bytes": by["layout"],
                       "gbs": round(by["layout"] / statistics.mean(lay_ms) / 1e6, 1)},
            "dispatch": {"ms": round(d_ms, 5), "bytes": by["dispatch"],
                         "gbs": round(by["dispatch"] / d_ms / 1e6, 1),
                         "frac_of_peak": round(by["dispatch"] / d_ms / 1e6 / peaks["hbm_gbs"], 4)},
            "combine": {"ms": round(c_ms, 5), "bytes": by["combine"],
                        "gbs": round(by["combine"] / c_ms / 1e6, 1),
                        "frac_of_peak": round(by["combine"] / c_ms / 1e6 / peaks["hbm_gbs"], 4)},
        },
        "layout_plus_dispatch_ms": round(statistics.mean(lay_ms) + d_ms, 5),
        "layout_host_ms": round(1e3 * statistics.median(layout_host_s), 5),
        "warm_l2": {"steps": warm_steps,
                    **{k: {"ms": round(v, 5), "gbs": round(by[k] / v / 1e6, 1)}
                       for k, v in warm.items()}},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "algorithmic_bytes": by[dom]},
        "e2e": {"value": round(total_bytes * ws / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5),
                "how": "C ABI with host buffers: per step, pinned h2d of topk_idx, weights and x, "
                       "layout + dispatch + combine, d2h of the output; consecutive steps "
                       "rotate over three streams, the next step's inputs are copied in before "
                       "this step's layout (copies overlap neighbouring steps)",
                "h2d_bytes_per_step": idx_h.numel() * 8 + w_h.numel() * 4 + x_h.numel() * 2,
                "d2h_bytes_per_step": T * H * 2},
        "gpu_launches": launches,
        "clocks": clk,
        "backward": {
            "steps": bwd_steps,
            "combine_backward": {"ms": round(cb_ms, 5), "bytes": bwd_by["combine_backward"],
                                 "gbs": round(bwd_by["combine_backward"] / cb_ms / 1e6, 1),
                                 "frac_of_peak": round(bwd_by["combine_backward"] / cb_ms / 1e6
                                                       / peaks["hbm_gbs"], 4)},
            "dispatch_backward": {"ms": round(db_ms, 5), "bytes": bwd_by["dispatch_backward"],
                                  "gbs": round(bwd_by["dispatch_backward"] / db_ms / 1e6, 1),
                                  "frac_of_peak": round(bwd_by["dispatch_backward"] / db_ms / 1e6
                                                        / peaks["hbm_gbs"], 4)},
            "gpu_launches": bwd_steps * ((1 if T > 0 else 0) + (2 if T > 0 else 0)),
        },
    }
    if pq is not None:
        pq["frac_of_peak"] = round(pq["gbs"] / peaks["hbm_gbs"], 4)
        line["dispatch_prequantised"] = pq
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cb = time_oracle(wl, args.cpu_sample_tokens, args.cpu_budget_s, seed=args.seed)
        line["cpu_baseline"] = {"value": round(cb["gbs"], 4), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": cb["sample"],
                                "tokens_per_s": round(cb["tokens_per_s"], 1),
                                "cpu_model": cpu_model()}
        allc = time_oracle_all_cores(wl, args.cpu_sample_tokens, args.cpu_budget_s, args.seed)
        if allc is not None:
            line["cpu_baseline_all_cores"] = allc
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, ws, rank):
    """The CPU oracle on the host cores: rank 0 only, bounded samples."""
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    torch.set_num_threads(1)   # the oracle is timed on one core; so is its setup
    # One calibration pass (it counts as a warm-up step) sizes the per-step
    # sample so the whole run stays near REFERENCE_BUDGET_S of CPU time.
    T = min(args.cpu_sample_tokens, wl.num_tokens)
    cal = time_oracle(wl, T, 0.0, seed=args.seed)
    per_step_s = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    if cal["sec_per_step"] > per_step_s:
        T = max(32, int(T * per_step_s / cal["sec_per_step"]) // 32 * 32)
    T, inp, y_bits = oracle_setup(wl, T, args.seed)
    per = []
    lay = None
    for i in range(max(0, args.warmup - 1) + args.steps):
        t0 = time.perf_counter()
        lay = oracle_step(wl, inp, y_bits)
        if i >= max(0, args.warmup - 1):
            per.append(time.perf_counter() - t0)
    sec = statistics.mean(per)
    total = sum(bytes_from_layout(wl, T, inp["topk_idx"], lay).values())
    res = {"gbs": total / sec / 1e9, "sec_per_step": sec,
           "sample": oracle_sample_text(wl, T, args.seed, len(per))}
    gbs = res["gbs"] * res["sec_per_step"] / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32", "data": "synthetic (seeded generators)",
        "config": {"workload": wl.name, "tokens": wl.num_tokens, "hidden": wl.hidden,
                   "sample_tokens_per_step": T},
        "tokens_per_s": round(T / sec, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": res["sample"]},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-sample-tokens", type=int, default=512)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_gpu(args, ws, rank, local)


if __name__ == "__main__":
    main()
