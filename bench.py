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
# Clock sampling: one nvidia-smi sampler across every GPU section of the run
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.sections = []      # (name, wall start, wall end)
        self.samples = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def section(self, name: str):
        """Context manager marking the wall-clock span of one GPU section."""
        sampler = self

        class _Span:
            def __enter__(self):
                torch.cuda.synchronize()
                self.t0 = time.time()

            def __exit__(self, *exc):
                torch.cuda.synchronize()
                sampler.sections.append((name, self.t0, time.time()))
        return _Span()

    def _parse(self, out: str):
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append({"t": ts + frac, "sm": float(f[2]), "smax": float(f[3]),
                             "power": float(f[4]),
                             "reasons": {n for n, v in zip(self.REASONS, f[6:10])
                                         if v.lower() == "active"}})
            except (ValueError, IndexError):
                continue
        return rows

    @staticmethod
    def _summary(rows) -> dict:
        if not rows:
            return {"sm_mhz": None, "samples": 0}
        sm = [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "samples": len(sm),
                "reasons": sorted(set().union(*[r["reasons"] for r in rows]))}

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = self._parse(out)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if any(a <= r["t"] <= b for _, a, b in self.sections)]
        use = inside or rows
        res = self._summary(use)
        res.update({"sm_max_mhz": max(r["smax"] for r in rows),
                    "power_w_max": max(r["power"] for r in use),
                    "period_ms": self.period_ms,
                    "over": "every measured GPU section" if inside else "the whole run",
                    "sections": {}})
        for name, a, b in self.sections:
            res["sections"][name] = self._summary([r for r in rows if a <= r["t"] <= b])
        return res


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
GATE_CYCLES = 2_000_000   # ~1 ms spin: the host enqueues the timed launches behind it
L2_BYTES = 126 << 20      # GB300 L2; inputs re-read by repeated launches rotate past it

# Kernels each stage launches (ours): layout = one cluster kernel or count +
# assign (the library reports which); dispatch = copy kernel (+ the
# column-major scale gather for FP8); combine = one kernel.
def launches(wl: W.Workload, rows_alloc: int, T: int, layout_kernels: int) -> dict:
    return {"layout": layout_kernels,
            "dispatch": (1 + int(wl.use_fp8 and wl.col_major_sf)) if rows_alloc > 0 else 0,
            "combine": 1 if T > 0 else 0}


class GpuWorkload:
    """One workload resident in HBM: inputs, the library config, expert
    outputs y for combine (identity experts: the dequantised or copied
    dispatch output, made once, untimed, by torch ops outside the path), the
    algorithmic bytes of each stage, and the timed loops."""

    def __init__(self, ep, wl: W.Workload, dev, seed: int, stream, flush_l2):
        self.ep, self.wl, self.dev, self.stream, self.flush_l2 = ep, wl, dev, stream, flush_l2
        T, H = wl.num_tokens, wl.hidden
        self.T, self.H = T, H
        inp = W.make_inputs(wl, seed=seed)
        self.idx_h, self.w_h, self.x_h = inp["topk_idx"], inp["topk_weights"], inp["x"]
        self.idx, self.w, self.x = self.idx_h.to(dev), self.w_h.to(dev), self.x_h.to(dev)
        self.eb = inp["expert_bias"].to(dev) if inp["expert_bias"] is not None else None
        self.cfg = ep.make_config(T, wl.num_topk, wl.num_experts, wl.num_ranks, H,
                                  wl.num_max_tokens_per_rank, wl.expert_alignment, wl.do_expand,
                                  wl.do_zero_padding, wl.do_cpu_sync, wl.use_fp8, wl.col_major_sf,
                                  fixed_capacity=wl.fixed_capacity)
        h0 = ep.ep_layout(self.cfg, self.idx)
        out0 = ep.alloc_recv(h0, with_weights=True, with_idx=True, zero=True)
        ep.ep_dispatch(h0, self.x, self.w, **out0)
        rows = h0.rows_alloc
        if wl.use_fp8:
            q = out0["recv_x"].view(torch.float8_e4m3fn).float()
            nb = H // 128
            sf = out0["recv_sf"]
            if wl.fixed_capacity and wl.col_major_sf:
                cap = wl.num_max_tokens_per_rank * wl.num_ranks
                st = -(-cap // 4) * 4
                s_ = sf.view(wl.num_experts, nb, st)[:, :, :cap].permute(0, 2, 1).reshape(rows, nb)
            elif wl.col_major_sf:
                s_ = sf.view(nb, -1)[:, :rows].t()
            else:
                s_ = sf.view(rows, nb)
            self.y = (q.view(rows, nb, 128) * s_.unsqueeze(-1)).view(rows, H).to(torch.bfloat16)
            del q
        else:
            self.y = out0["recv_x"].clone()
        g0 = {n: h0.tensor(n).cpu() for n in ("dst_buffer_slot_idx", "cnt_expert",
                                                "cnt_expert_aligned", "totals")}
        torch.cuda.synchronize()
        dst = g0["dst_buffer_slot_idx"]
        self.pad_rows = int((g0["cnt_expert_aligned"] - g0["cnt_expert"]).sum()) \
            if wl.do_expand else 0
        total_rows = int(g0["totals"][1] if wl.do_expand else g0["totals"][0])
        self.valid_rows = total_rows - self.pad_rows
        self.distinct = int(torch.unique(dst[dst >= 0]).numel())
        self.by = stage_bytes(wl, T, self.idx_h, self.valid_rows, self.pad_rows, self.distinct,
                              expert_bias=self.eb is not None)
        self.out_comb = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.grad_recv_w = out0["recv_topk_weights"].clone()
        self.rows_alloc = rows
        self.n_launch = launches(wl, rows, T, int(h0.info.layout_kernels))
        h0.free()
        del out0

    def _gate(self):
        torch.cuda._sleep(GATE_CYCLES)

    def step(self, ev=None):
        """One back-to-back step: layout -> dispatch -> combine, nothing
        between them on the device, every launch enqueued behind a spin
        kernel so no host code runs inside a timed interval.  ev (4 events):
        without the count wait one interval [ev0, ev3] covers the step, with
        no event between the kernels (so each may start while the one before
        it drains, as the kernels are launched), layout and dispatch by one
        ep_layout_dispatch call into buffers sized from the configuration;
        with it the layout interval [ev0, ev1] includes the host's reaction
        to the counts (as for every caller of the exact allocation), and
        [ev2, ev3] covers dispatch and combine, enqueued behind a second spin
        kernel."""
        ep, sync = self.ep, bool(self.cfg.do_cpu_sync)
        if not sync:  # host-side allocation (torch's caching allocator), before the gate
            out = ep.alloc_recv_planned(self.cfg, with_weights=True, with_idx=True)
        self._gate()
        if ev:
            ev[0].record(self.stream)
        if sync:
            h = ep.ep_layout(self.cfg, self.idx)
            if ev:
                ev[1].record(self.stream)
            out = ep.alloc_recv(h, with_weights=True, with_idx=True)
            self._gate()
            if ev:
                ev[2].record(self.stream)
            ep.ep_dispatch(h, self.x, self.w, **out)
        else:
            h = ep.ep_layout_dispatch(self.cfg, self.idx, self.x, self.w, **out)
        ep.ep_combine(h, self.y, self.w, None, None, self.eb, out=self.out_comb)
        if ev:
            ev[3].record(self.stream)
        h.free()

    def step_time(self, ev) -> float:
        if self.cfg.do_cpu_sync:
            return ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3])
        return ev[0].elapsed_time(ev[3])

    def step_staged(self, ev=None):
        """The back-to-back step with an event between consecutive stages, for
        the per-stage breakdown (the events keep each kernel from starting
        before the one before it has ended).  ev (5 events): layout start /
        end, dispatch start, dispatch end = combine start, combine end."""
        ep, sync = self.ep, bool(self.cfg.do_cpu_sync)
        self._gate()
        if ev:
            ev[0].record(self.stream)
        h = ep.ep_layout(self.cfg, self.idx)
        if ev:
            ev[1].record(self.stream)
        out = ep.alloc_recv(h, with_weights=True, with_idx=True)
        if sync:
            self._gate()
        if ev:
            ev[2].record(self.stream)
        ep.ep_dispatch(h, self.x, self.w, **out)
        if ev:
            ev[3].record(self.stream)
        ep.ep_combine(h, self.y, self.w, None, None, self.eb, out=self.out_comb)
        if ev:
            ev[4].record(self.stream)
        h.free()

    def step_flushed(self, ev=None):
        """The same step with an L2 flush (untimed) before every stage: each
        stage starts from a cold L2 holding no dirty lines, so the write-back
        of what a stage leaves dirty falls in the next, untimed flush."""
        ep = self.ep
        self.flush_l2()
        if ev:
            ev[0].record(self.stream)
        h = ep.ep_layout(self.cfg, self.idx)
        if ev:
            ev[1].record(self.stream)
        out = ep.alloc_recv(h, with_weights=True, with_idx=True)
        self.flush_l2()
        if ev:
            ev[2].record(self.stream)
        ep.ep_dispatch(h, self.x, self.w, **out)
        if ev:
            ev[3].record(self.stream)
        self.flush_l2()
        if ev:
            ev[4].record(self.stream)
        ep.ep_combine(h, self.y, self.w, None, None, self.eb, out=self.out_comb)
        if ev:
            ev[5].record(self.stream)
        h.free()

    def run_whole_steps(self, n: int, warmup: int) -> float:
        """Warm-up, then n back-to-back steps with the L2 flushed between
        steps; returns the mean step time (ms)."""
        for _ in range(warmup):
            self.flush_l2()
            self.step()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for i in range(n):
            self.flush_l2()
            self.step(evs[i])
        torch.cuda.synchronize()
        return statistics.mean(self.step_time(e) for e in evs)

    def run_steps(self, n: int, warmup: int, flushed: bool = False) -> dict:
        """Warm-up, then n staged steps with the L2 flushed between steps;
        returns the mean per-stage device times (ms)."""
        fn = self.step_flushed if flushed else self.step_staged
        for _ in range(warmup):
            if not flushed:
                self.flush_l2()
            fn()
        torch.cuda.synchronize()
        nev = 6 if flushed else 5
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(n)]
        for i in range(n):
            if not flushed:
                self.flush_l2()
            fn(evs[i])
        torch.cuda.synchronize()
        if flushed:
            lay = [e[0].elapsed_time(e[1]) for e in evs]
            dis = [e[2].elapsed_time(e[3]) for e in evs]
            com = [e[4].elapsed_time(e[5]) for e in evs]
        else:
            lay = [e[0].elapsed_time(e[1]) for e in evs]
            dis = [e[2].elapsed_time(e[3]) for e in evs]
            com = [e[3].elapsed_time(e[4]) for e in evs]
        return {"layout": statistics.mean(lay), "dispatch": statistics.mean(dis),
                "combine": statistics.mean(com),
                "step": statistics.mean(a + b + c for a, b, c in zip(lay, dis, com)),
                "launches": n * sum(self.n_launch.values())}

    def stage_block(self, t: dict, peak: float) -> dict:
        out = {}
        for k in ("layout", "dispatch", "combine"):
            gbs = self.by[k] / t[k] / 1e6
            out[k] = {"ms": round(t[k], 5), "bytes": self.by[k], "gbs": round(gbs, 1)}
            if k != "layout":
                out[k]["frac_of_peak"] = round(gbs / peak, 4)
        tot = sum(self.by.values())
        out["step"] = {"ms": round(t["step"], 5), "bytes": tot,
                       "gbs": round(tot / t["step"] / 1e6, 1),
                       "frac_of_peak": round(tot / t["step"] / 1e6 / peak, 4),
                       "tokens_per_s": round(self.T / (t["step"] * 1e-3), 1)}
        return out

    def _copies(self, t: torch.Tensor) -> list:
        """t and enough clones that cycling through them re-reads more than
        twice the L2 between two uses of one copy."""
        n = max(1, min(4, -(-2 * L2_BYTES // max(1, t.numel() * t.element_size()))))
        return [t] + [t.clone() for _ in range(n - 1)]

    def soak(self, seconds: float, peak: float) -> dict:
        """Dispatch + combine pairs launched back to back for about `seconds`
        (inputs rotating over copies larger than L2); throughput over the
        whole run, which reaches the power and thermal steady state."""
        ep = self.ep
        h = ep.ep_layout(self.cfg, self.idx)
        out = ep.alloc_recv(h, with_weights=True, with_idx=True)
        xs, ys = self._copies(self.x), self._copies(self.y)

        def pair(i):
            ep.ep_dispatch(h, xs[i % len(xs)], self.w, **out)
            ep.ep_combine(h, ys[i % len(ys)], self.w, None, None, self.eb, out=self.out_comb)

        for i in range(3):
            pair(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pair(0)
        torch.cuda.synchronize()
        one = max(time.perf_counter() - t0, 1e-5)
        n = max(10, int(seconds / one))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self._gate()
        e0.record(self.stream)
        for i in range(n):
            pair(i)
        e1.record(self.stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        by = self.by["dispatch"] + self.by["combine"]
        gbs = by * n / (ms * 1e-3) / 1e9
        h.free()
        return {"pairs": n, "seconds": round(ms * 1e-3, 3), "gbs": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4), "gpu_launches": n * (
                    self.n_launch["dispatch"] + self.n_launch["combine"])}

    def sustained(self, n: int, peak: float) -> dict:
        """Dispatch alone, then combine alone, launched n times back to back
        behind a spin kernel: each launch pays the write-back of the lines the
        launch before it left dirty, i.e. in steady state its own.  Inputs
        rotate over copies that together exceed the L2."""
        ep = self.ep
        h = ep.ep_layout(self.cfg, self.idx)
        out = ep.alloc_recv(h, with_weights=True, with_idx=True)
        xs = self._copies(self.x)
        ys = self._copies(self.y)
        res = {}
        for name in ("dispatch", "combine"):
            def launch(i):
                if name == "dispatch":
                    ep.ep_dispatch(h, xs[i % len(xs)], self.w, **out)
                else:
                    ep.ep_combine(h, ys[i % len(ys)], self.w, None, None, self.eb,
                                  out=self.out_comb)
            for i in range(3):
                launch(i)
            self.flush_l2()
            self._gate()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for i in range(n):
                launch(i)
            e1.record(self.stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            gbs = self.by[name] / ms / 1e6
            res[name] = {"ms": round(ms, 5), "gbs": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4), "launches": n,
                         "input_copies": len(xs) if name == "dispatch" else len(ys)}
        h.free()
        del xs, ys
        return res


def run_gpu(args, ws, rank, local):
    import combine_topk_idx_gb300 as ep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    ep.load_library()
    peaks = load_peaks()
    peak = peaks["hbm_gbs"]
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one, so that the
        # next timed launch starts with a cold L2 holding no dirty lines
        flush_w.zero_()
        flush_r.sum()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    wl = W.WORKLOADS[args.workload]
    main = GpuWorkload(ep, wl, dev, args.seed, stream, flush_l2)
    T, H = main.T, main.H
    by = main.by
    total_bytes = sum(by.values())

    # ---- the timed steps: back to back, L2 flushed between steps ----
    for _ in range(args.warmup):
        flush_l2()
        main.step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(ws)
    with clocks.section("timed_steps"):
        for i in range(args.steps):
            flush_l2()
            main.step(evs[i])
    barrier(ws)
    step_ms = statistics.mean(main.step_time(e) for e in evs)
    step_ms_max = max_over_ranks(step_ms, ws, dev)
    value = total_bytes * ws / (step_ms_max * 1e-3) / 1e9
    n_launch = args.steps * sum(main.n_launch.values())

    # ---- secondary figures on the same workload ----
    # per-stage breakdown of the same step (an event between stages)
    fl_steps = max(8, args.steps // 2)
    with clocks.section("stages_staged"):
        t_main = main.run_steps(fl_steps, 3)
    with clocks.section("stages_flushed"):
        t_fl = main.run_steps(fl_steps, 3, flushed=True)
    with clocks.section("sustained"):
        sus = main.sustained(max(10, args.steps // 2), peak)
    # Soak: dispatch and combine back to back for about args.soak_s seconds
    # (power and thermal steady state); most clock samples come from here.
    soak = None
    if args.soak_s > 0:
        with clocks.section("soak"):
            soak = main.soak(args.soak_s, peak)
    # Host wall time of the layout call on an idle GPU (with do_cpu_sync it
    # includes the count wait).
    layout_host_s = []
    with clocks.section("layout_host"):
        for _ in range(20):
            torch.cuda.synchronize()
            t_host = time.perf_counter()
            h = ep.ep_layout(main.cfg, main.idx)
            layout_host_s.append(time.perf_counter() - t_host)
            h.free()

    # e2e through the C ABI with host buffers: every step copies its inputs
    # (topk_idx, topk_weights, x) in from pinned host memory and its combined
    # output back out.  Steps rotate over three streams and buffer sets, and
    # the next step's input copies are enqueued before this step's layout
    # (whose count wait blocks the host), so one step's copies overlap the
    # neighbouring steps' kernels and copies, as a serving loop would run them.
    idx_pin, w_pin, x_pin = main.idx_h.pin_memory(), main.w_h.pin_memory(), main.x_h.pin_memory()
    nbuf = 3
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(nbuf)]
    e2e_bufs = [{"idx": torch.empty_like(main.idx), "w": torch.empty_like(main.w),
                 "x": torch.empty_like(main.x),
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
            h = ep.ep_layout(main.cfg, b["idx"], stream=st)
            out = ep.alloc_recv(h, with_weights=True, with_idx=True)
            ep.ep_dispatch(h, b["x"], b["w"], **out, stream=st)
            ep.ep_combine(h, main.y, b["w"], None, None, main.eb, out=b["out"], stream=st)
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
    with clocks.section("e2e"):
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush_l2()
        e_s.record(stream)
        e2e_run(e2e_steps)
        e_e.record(stream)
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, ws, dev)
    barrier(ws)

    # Backward pair on one handle (layout untimed): combine_backward dispatches
    # a [T, H] gradient, dispatch_backward combines a [rows, H] gradient and
    # reduces the weight gradients.  L2 is flushed before each timed call.
    bwd_by = backward_bytes(wl, T, main.idx_h, main.valid_rows, main.pad_rows, main.distinct)
    hb = ep.ep_layout(main.cfg, main.idx)
    g_recv = torch.empty((hb.rows_alloc, H), dtype=torch.bfloat16, device=dev)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    g_w = torch.empty((T, wl.num_topk), dtype=torch.float32, device=dev)

    def bwd_step(ev=None):
        flush_l2()
        if ev:
            ev[0].record(stream)
        ep.ep_combine_backward(hb, main.x, g_recv)
        if ev:
            ev[1].record(stream)
        flush_l2()
        if ev:
            ev[2].record(stream)
        ep.ep_dispatch_backward(hb, main.y, main.grad_recv_w, g_x, g_w)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        bwd_step()
    bwd_steps = max(8, args.steps // 4)
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(bwd_steps)]
    with clocks.section("backward"):
        for i in range(bwd_steps):
            bwd_step(bev[i])
    cb_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in bev)
    db_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in bev)
    del g_recv, g_x, g_w

    # Dispatch of a pre-quantised input (FP8 workloads): x as e4m3 bytes with
    # column-major TMA-aligned fp32 scales, made once by torch, untimed.
    pq = None
    if wl.use_fp8:
        nb = H // 128
        xb = main.x.float().view(T, nb, 128)
        sc = xb.abs().amax(-1) / 448.0
        sc = torch.where(sc > 0, sc, torch.ones_like(sc))
        xq = (xb / sc.unsqueeze(-1)).to(torch.float8_e4m3fn).view(T, H)
        st = -(-max(T, 1) // 4) * 4
        sf_store = torch.zeros((nb, st), dtype=torch.float32, device=dev)
        sf_store[:, :T] = sc.t()
        xs = sf_store[:, :T].t()
        del xb
        pq_out = ep.alloc_recv(hb, with_weights=True, with_idx=True)
        pq_by = prequantised_bytes(wl, T, main.idx_h, main.valid_rows, main.pad_rows)

        def pq_step(ev=None):
            flush_l2()
            if ev:
                ev[0].record(stream)
            ep.ep_dispatch_fp8(hb, xq, xs, main.w, **pq_out)
            if ev:
                ev[1].record(stream)

        for _ in range(args.warmup):
            pq_step()
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(bwd_steps)]
        with clocks.section("dispatch_prequantised"):
            for i in range(bwd_steps):
                pq_step(pev[i])
        pq_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in pev)
        pq = {"steps": bwd_steps, "ms": round(pq_ms, 5), "bytes": pq_by,
              "gbs": round(pq_by / pq_ms / 1e6, 1),
              "frac_of_peak": round(pq_by / pq_ms / 1e6 / peak, 4),
              "input_sf": "column-major TMA-aligned", "l2": "flushed before each call",
              "gpu_launches": bwd_steps * (1 + int(wl.col_major_sf))}
        del pq_out, xq, sf_store
    hb.free()

    # ---- every other workload: the same back-to-back step and the flushed
    # stages, a few steps each (N = 1 only) ----
    wl_block = {}
    if ws == 1 and not args.no_workloads:
        del main.y
        for name in [n for n in ("decode", "decode_ll", "skewed", "large", "tiny")
                     if n != wl.name]:
            other = GpuWorkload(ep, W.WORKLOADS[name], dev, args.seed, stream, flush_l2)
            with clocks.section(f"workload_{name}"):
                tw = other.run_whole_steps(args.workload_steps, 3)
                tb = other.run_steps(args.workload_steps, 3)
                tf = other.run_steps(args.workload_steps, 3, flushed=True)
                su = other.sustained(args.workload_steps, peak)
            whole = sum(other.by.values())
            wl_block[name] = {
                "config": {"tokens": other.T, "hidden": other.H,
                           "experts": other.wl.num_experts,
                           "logical_ranks": other.wl.num_ranks, "topk": other.wl.num_topk,
                           "do_expand": other.wl.do_expand, "fp8_dispatch": other.wl.use_fp8,
                           "do_cpu_sync": other.wl.do_cpu_sync,
                           "fixed_capacity": other.wl.fixed_capacity},
                "steps": args.workload_steps,
                "step": {"ms": round(tw, 5), "bytes": whole,
                         "gbs": round(whole / tw / 1e6, 1),
                         "frac_of_peak": round(whole / tw / 1e6 / peak, 4),
                         "tokens_per_s": round(other.T / (tw * 1e-3), 1),
                         "calls": ("ep_layout (count wait), ep_dispatch, ep_combine"
                                   if other.wl.do_cpu_sync else
                                   "ep_layout_dispatch, ep_combine")},
                "back_to_back": other.stage_block(tb, peak),
                "stages_flushed": other.stage_block(tf, peak),
                "sustained": su,
                "gpu_launches": tb["launches"] + tf["launches"],
            }
            del other
            torch.cuda.empty_cache()

    clk = clocks.stop()
    d_ms, c_ms = t_main["dispatch"], t_main["combine"]
    dom = "combine" if c_ms >= d_ms else "dispatch"
    dom_ms = c_ms if dom == "combine" else d_ms
    achieved = by[dom] / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(dom, wl.name)
    stages = main.stage_block(t_main, peak)
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
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read); inside a "
                         "step the stages run back to back; times are device events",
                   "parallelism": f"replicas x{ws}"},
        "tokens_per_s": round(T * ws / (step_ms_max * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * value / ws / peak, 2),
        "step_how": "one step = layout, dispatch, combine back to back on the device, "
                    "launches enqueued behind a spin kernel so no host code falls inside the "
                    "timed intervals: the layout interval (it includes the host's reaction to "
                    "the count wait) plus one interval over dispatch and combine, with no "
                    "event between the kernels",
        "stages": {**{k: v for k, v in stages.items() if k != "step"},
                   "staged_step_ms": round(t_main["step"], 5), "steps": fl_steps},
        "stages_how": "the same step with an event between consecutive stages (each kernel "
                      "then starts only after the one before it has ended): per-stage device "
                      "times",
        "layout_plus_dispatch_ms": round(t_main["layout"] + d_ms, 5),
        "layout_host_ms": round(1e3 * statistics.median(layout_host_s), 5),
        "stages_flushed": {**{k: v for k, v in main.stage_block(t_fl, peak).items()},
                           "steps": fl_steps,
                           "how": "L2 flushed before every stage (no dirty lines inherited; "
                                  "a stage's own dirty lines drain in the next, untimed flush)"},
        "sustained": {**sus, "how": "each kernel launched back to back behind a spin kernel, "
                                    "inputs rotating over copies larger than L2: every launch "
                                    "pays the write-back of its predecessor's dirty lines, in "
                                    "steady state its own"},
        "soak": soak,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": by[dom],
                     "sustained_frac": sus[dom]["frac_of_peak"]},
        "e2e": {"value": round(total_bytes * ws / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5),
                "how": "C ABI with host buffers: per step, pinned h2d of topk_idx, weights and x, "
                       "layout + dispatch + combine, d2h of the output; consecutive steps "
                       "rotate over three streams, the next step's inputs are copied in before "
                       "this step's layout (copies overlap neighbouring steps)",
                "h2d_bytes_per_step": main.idx_h.numel() * 8 + main.w_h.numel() * 4
                + main.x_h.numel() * 2,
                "d2h_bytes_per_step": T * H * 2},
        "gpu_launches": n_launch,
        "clocks": clk,
        "backward": {
            "steps": bwd_steps, "l2": "flushed before each call",
            "combine_backward": {"ms": round(cb_ms, 5), "bytes": bwd_by["combine_backward"],
                                 "gbs": round(bwd_by["combine_backward"] / cb_ms / 1e6, 1),
                                 "frac_of_peak": round(bwd_by["combine_backward"] / cb_ms / 1e6
                                                       / peak, 4)},
            "dispatch_backward": {"ms": round(db_ms, 5), "bytes": bwd_by["dispatch_backward"],
                                  "gbs": round(bwd_by["dispatch_backward"] / db_ms / 1e6, 1),
                                  "frac_of_peak": round(bwd_by["dispatch_backward"] / db_ms / 1e6
                                                        / peak, 4)},
            "gpu_launches": bwd_steps * ((1 if T > 0 else 0) + (2 if T > 0 else 0)),
        },
    }
    if pq is not None:
        line["dispatch_prequantised"] = pq
    if wl_block:
        line["workloads"] = wl_block
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


def run_stage(args):
    """One stage of one workload launched --stage-launches times through the C
    ABI, L2 flushed (256 MiB write + 256 MiB read) before each launch; prints
    the mean device time.  Meant for profiling a single kernel (ncu -k ... -s
    ... -c ...); the step benchmark above is the measurement."""
    import combine_topk_idx_gb300 as ep
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ep.load_library()
    wl = W.WORKLOADS[args.workload]
    inp = W.make_inputs(wl, seed=args.seed)
    idx, w, x = inp["topk_idx"].to(dev), inp["topk_weights"].to(dev), inp["x"].to(dev)
    eb = inp["expert_bias"].to(dev) if inp["expert_bias"] is not None else None
    cfg = ep.make_config(wl.num_tokens, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden,
                         wl.num_max_tokens_per_rank, wl.expert_alignment, wl.do_expand,
                         wl.do_zero_padding, wl.do_cpu_sync, wl.use_fp8, wl.col_major_sf,
                         fixed_capacity=wl.fixed_capacity)
    h = ep.ep_layout(cfg, idx)
    out = ep.alloc_recv(h, with_weights=True, with_idx=True)
    y = W.make_bf16_rows(h.rows_alloc, wl.hidden, args.seed).to(dev)
    res = torch.empty((wl.num_tokens, wl.hidden), dtype=torch.bfloat16, device=dev)
    g_recv = torch.empty((h.rows_alloc, wl.hidden), dtype=torch.bfloat16, device=dev)
    g_w = torch.empty((wl.num_tokens, wl.num_topk), dtype=torch.float32, device=dev)
    grad_recv_w = torch.zeros(out["recv_topk_weights"].shape, dtype=torch.float32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def launch():
        if args.stage == "layout":
            ep.ep_layout(cfg, idx).free()
        elif args.stage == "dispatch":
            ep.ep_dispatch(h, x, w, **out)
        elif args.stage == "combine":
            ep.ep_combine(h, y, w, None, None, eb, out=res)
        elif args.stage == "combine_backward":
            ep.ep_combine_backward(h, x, g_recv)
        else:  # dispatch_backward
            ep.ep_dispatch_backward(h, y, grad_recv_w, res, g_w)

    ms = []
    for _ in range(args.stage_launches):
        flush_w.zero_()
        flush_r.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        launch()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    h.free()
    print(json.dumps({"stage": args.stage, "workload": wl.name, "launches": len(ms),
                      "ms_mean": round(statistics.mean(ms), 5),
                      "l2": "flushed before each launch"}), flush=True)


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
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the block that times every other workload")
    ap.add_argument("--workload-steps", type=int, default=10)
    ap.add_argument("--stage", choices=["layout", "dispatch", "combine", "combine_backward",
                                        "dispatch_backward"],
                    help="launch one stage only (for profiling one kernel)")
    ap.add_argument("--stage-launches", type=int, default=4)
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="seconds of back-to-back dispatch + combine at the end (0: none)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.stage:
        run_stage(args)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_gpu(args, ws, rank, local)


if __name__ == "__main__":
    main()
