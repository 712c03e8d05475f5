"""GPU parity of the fixed-capacity per-expert layout (DeepEP README,
"Interfaces and examples", low_latency_dispatch / low_latency_combine: a
per-rank [local experts, max tokens per rank * ranks, hidden] receive tensor
with per-expert counts, usable under CUDA graphs) against the oracle.

Layout, metadata, payload, scales (per-expert column-major slabs or
row-major), weights bit-exact; combine within 1 BF16 ulp.  The same handle
also drives the backward pair and the pre-quantised dispatch.
"""
import zlib

import numpy as np
import pytest
import torch

import ep_workloads as W
from oracle import ep_oracle as O
from tests import ep_harness as HN
from tests.test_backward_gpu import check_backward
from tests.test_parity_gpu import make_y, run_and_check
from tests.test_prequant_gpu import run_prequant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def _routing(T, K, E, seed, drop=0.0, dup=False):
    g = torch.Generator().manual_seed(seed)
    if dup:
        idx = torch.randint(0, E, (T, K), generator=g)
    else:
        idx = torch.rand(T, E, generator=g).topk(min(K, E), dim=1).indices
    if drop > 0:
        idx = idx.masked_fill(torch.rand(T, K, generator=g) < drop, -1)
    w = torch.rand(T, K, generator=g).masked_fill(idx < 0, 0.0)
    return idx.to(torch.int64).contiguous(), w.contiguous()


def fixed_cfg(ep, T, K, E, R, H, M, sync, fp8, cm):
    return ep.make_config(T, K, E, R, H, M, 1, True, False, sync, fp8, cm, fixed_capacity=True)


CASES = {
    # name: (T, K, E, R, H, M, sync, fp8, col_major, drop, dup)
    "decode_like_fp8_cm": (512, 8, 64, 8, 1024, 64, False, True, True, 0.0, False),
    "fp8_rowmajor_sync": (300, 6, 32, 4, 256, 75, True, True, False, 0.1, False),
    "bf16_nosync": (333, 4, 16, 4, 8 * 37, 100, False, False, False, 0.1, False),
    "fp8_cm_odd_capacity": (45, 3, 12, 3, 384, 15, False, True, True, 0.0, False),
    "repeated_experts_overflow": (8, 4, 4, 2, 128, 4, False, True, True, 0.0, True),
    "all_slots_empty": (40, 3, 8, 4, 128, 10, False, True, True, 1.0, False),
    "empty_tokens": (0, 4, 8, 2, 128, 4, False, True, True, 0.0, False),
    "one_rank": (200, 2, 6, 1, 128, 200, True, False, False, 0.0, False),
    # many layout chunks (32 and 20 source ranks; expanded layouts always take
    # the count + assign kernels)
    "many_chunks_fp8_cm": (1000, 6, 64, 32, 256, 32, False, True, True, 0.05, False),
    "many_chunks_overflow": (40, 4, 20, 20, 128, 2, True, True, False, 0.0, True),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fixed_capacity_parity(ep, case):
    T, K, E, R, H, M, sync, fp8, cm, drop, dup = CASES[case]
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop, dup=dup)
    if dup:
        idx[:, :2] = 0      # expert 0 named twice by every token: past its capacity
    cfg = fixed_cfg(ep, T, K, E, R, H, M, sync, fp8, cm)
    r = run_and_check(ep, cfg, idx, torch.randn(T, H).to(torch.bfloat16), w, bias0=True)
    lay = r["lay"]
    assert lay["rows_alloc"] == E * M * R
    if dup:
        assert lay["error"] & 2
    assert r["combine_mismatch"] == 0


def test_fixed_capacity_handle_reports_strides(ep):
    T, K, E, R, H, M = 64, 4, 16, 4, 512, 16
    idx, _ = _routing(T, K, E, seed=5)
    for cm in (True, False):
        cfg = fixed_cfg(ep, T, K, E, R, H, M, False, True, cm)
        h = ep.ep_layout(cfg, idx.cuda())
        cap = M * R
        nb = H // 128
        assert h.info.expert_capacity == cap and h.rows_alloc == E * cap
        if cm:
            cap_al = -(-cap // 4) * 4
            assert (h.info.sf_token_stride, h.info.sf_hidden_stride) == (1, cap_al)
            assert h.info.sf_expert_stride == nb * cap_al
        else:
            assert (h.info.sf_token_stride, h.info.sf_hidden_stride) == (nb, 1)
            assert h.info.sf_expert_stride == nb * cap
        assert h.info.sf_numel == O.sf_numel(E * cap, H, cm, cap)
        torch.cuda.synchronize()
        h.free()


@pytest.mark.parametrize("cm_in", [False, True])
def test_fixed_capacity_prequantised(ep, cm_in):
    T, K, E, R, H, M = 256, 8, 32, 4, 512, 64
    idx, w = _routing(T, K, E, seed=9, drop=0.05)
    cfg = fixed_cfg(ep, T, K, E, R, H, M, False, True, True)
    run_prequant(ep, cfg, idx, w, cm_in)


def test_fixed_capacity_backward_pair(ep):
    T, K, E, R, H, M = 256, 8, 32, 4, 256, 64
    idx, _ = _routing(T, K, E, seed=11, drop=0.05)
    cfg = fixed_cfg(ep, T, K, E, R, H, M, False, True, True)
    assert check_backward(ep, cfg, idx) == 0


def test_fixed_capacity_cuda_graph_replay(ep):
    """The fixed layout has static shapes: capture layout + dispatch + combine
    (+ handle free) once, replay on new routing and inputs, and compare the
    payload, scales, weights and combined output of every replay with the
    oracle."""
    T, K, E, R, H, M = 512, 8, 64, 8, 512, 64
    cfg = fixed_cfg(ep, T, K, E, R, H, M, False, True, True)
    rows = ep.upper_bound_rows(cfg)
    dev = torch.device("cuda")
    idx_s = torch.empty((T, K), dtype=torch.int64, device=dev)
    w_s = torch.empty((T, K), dtype=torch.float32, device=dev)
    x_s = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    y_s = make_y(rows, H, 31, dev)
    cap = M * R
    sfn = O.sf_numel(rows, H, True, cap)
    recv = {"recv_x": torch.zeros((rows, H), dtype=torch.uint8, device=dev),
            "recv_sf": torch.zeros((sfn,), dtype=torch.float32, device=dev),
            "recv_topk_weights": torch.zeros((rows,), dtype=torch.float32, device=dev)}
    res = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def path(st):
        h = ep.ep_layout(cfg, idx_s, stream=st)
        ep.ep_dispatch(h, x_s, w_s, stream=st, **recv)
        ep.ep_combine(h, y_s, w_s, out=res, stream=st)
        h.free()

    def fill(seed):
        idx, w = _routing(T, K, E, seed=seed, drop=0.05)
        idx_s.copy_(idx)
        w_s.copy_(w)
        x_s.copy_(torch.randn(T, H, generator=torch.Generator().manual_seed(seed))
                  .to(torch.bfloat16))
        return idx, w

    s = torch.cuda.Stream()
    fill(0)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        path(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        path(s)
    for seed in (3, 4):
        idx, w = fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        lay = HN.oracle_layout(cfg, idx.numpy())
        d_or = O.dispatch(lay, HN.bits16(x_s), w.numpy(), True, True, False)
        pdef = d_or["payload_defined"]
        assert np.array_equal(recv["recv_x"].cpu().numpy()[pdef], d_or["recv_x"][pdef])
        gs = recv["recv_sf"].cpu().numpy()
        rws = np.flatnonzero(pdef)
        for j in range(H // 128):
            ix = O.sf_index(rws, j, rows, H, True, cap)
            assert np.array_equal(gs[ix], d_or["recv_sf"][ix])
        assert np.array_equal(recv["recv_topk_weights"].cpu().numpy()[pdef],
                              d_or["recv_topk_weights"][pdef])
        need = np.flatnonzero(pdef)
        y_bits = np.zeros((rows, H), dtype=np.uint16)
        y_bits[need] = HN.bits16(W.hashed_bf16_rows(torch.from_numpy(need), H, 31))
        ref = O.combine(lay, y_bits, w.numpy())
        d = HN.ulp_diff(HN.bits16(res), ref)
        assert d.max(initial=0) <= 1
