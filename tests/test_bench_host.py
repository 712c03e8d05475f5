"""Host logic of bench.py: byte accounting, replica aggregation over ranks
(two gloo processes on the CPU), the committed-traffic lookup, and the
reference arm (the oracle) on a tiny sample."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import ep_workloads as W
from oracle import ep_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r, _ = bench.dist_env()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    mx = bench.max_over_ranks(10.0 + 5 * r, ws)
    sm = bench.sum_over_ranks(1.0 + r, ws)
    bench.barrier(ws)
    dist.destroy_process_group()
    out_q.put((r, mx, sm))


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [x[1] for x in res] == [15.0, 15.0]        # max over ranks, seen by every rank
    assert [x[2] for x in res] == [3.0, 3.0]


def test_single_rank_helpers_are_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(2.0, 1) == 2.0


def test_stage_bytes_match_definition():
    wl = W.WORKLOADS["tiny"]
    idx, w = W.make_routing(wl, seed=0)
    lay = O.layout(idx.numpy(), wl.num_experts, wl.num_ranks, wl.num_max_tokens_per_rank,
                   wl.expert_alignment, wl.do_expand, True)
    by = bench.bytes_from_layout(wl, wl.num_tokens, idx, lay)
    T, K, H, R = wl.num_tokens, wl.num_topk, wl.hidden, wl.num_ranks
    valid = (idx >= 0).numpy()
    rows = int(valid.sum())
    pad = int((lay["cnt_expert_aligned"] - lay["cnt_expert"]).sum())
    act = int(valid.any(axis=1).sum())
    assert by["layout"] == T * K * 16 + rows * 8 + T * R
    assert by["dispatch"] == act * H * 2 + T * K * 12 + rows * (2 * H + 4) + pad * (2 * H + 4)
    assert by["combine"] == rows * H * 2 + T * K * 8 + T * H * 2


def test_recorded_traffic_lookup(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "combine_topk_idx_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "ep_combine.cu").write_text("kernel v1")
    h = bench.kernel_source_hash("ep_combine.cu")
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        f"# kernel workload bytes source-hash\ncombine prefill 123456 {h}\n")
    assert bench.recorded_traffic("combine", "prefill") == 123456
    assert bench.recorded_traffic("combine", "large") is None
    (csrc / "ep_combine.cu").write_text("kernel v2")      # source changed since the capture
    assert bench.recorded_traffic("combine", "prefill") is None


def test_reference_arm_runs_the_oracle():
    env = dict(os.environ, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3",
                          "--cpu-sample-tokens", "64"], capture_output=True, text=True,
                         env=env, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # other ranks of a multi-rank launch print nothing
    env2 = dict(env, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, env=env2, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_backward_bytes_match_definition():
    for name in ("tiny", "decode"):
        wl = W.WORKLOADS[name]
        idx, _ = W.make_routing(wl, seed=0)
        lay = O.layout(idx.numpy(), wl.num_experts, wl.num_ranks, wl.num_max_tokens_per_rank,
                       wl.expert_alignment, wl.do_expand, True)
        T, K, H = wl.num_tokens, wl.num_topk, wl.hidden
        valid = (idx >= 0).numpy()
        dst = lay["dst_buffer_slot_idx"]
        distinct = int(np.unique(dst[dst >= 0]).size)
        pad = int((lay["cnt_expert_aligned"] - lay["cnt_expert"]).sum()) if wl.do_expand else 0
        rows = distinct
        by = bench.backward_bytes(wl, T, idx, rows, pad, distinct)
        act = int(valid.any(axis=1).sum())
        zp = wl.do_expand and wl.do_zero_padding
        assert by["combine_backward"] == act * H * 2 + T * K * 8 + rows * 2 * H + (pad * 2 * H if zp else 0)
        g = 4 if wl.do_expand else 4 * K
        assert by["dispatch_backward"] == distinct * 2 * H + T * K * 12 + T * H * 2 + rows * g


def test_prequantised_bytes_match_definition():
    wl = W.WORKLOADS["prefill"]
    T = 256
    idx, _ = W.make_routing(wl, seed=0, num_tokens=T)
    lay = O.layout(idx.numpy(), wl.num_experts, wl.num_ranks, wl.num_max_tokens_per_rank,
                   wl.expert_alignment, wl.do_expand, True)
    valid = (idx >= 0).numpy()
    rows = int(valid.sum())
    pad = int((lay["cnt_expert_aligned"] - lay["cnt_expert"]).sum())
    act = int(valid.any(axis=1).sum())
    H, K = wl.hidden, wl.num_topk
    sf = H // 128 * 4
    assert bench.prequantised_bytes(wl, T, idx, rows, pad) == \
        act * (H + sf) + T * K * 12 + rows * (H + sf + 4) + pad * (H + sf + 4)
