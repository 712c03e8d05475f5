"""GPU parity of ep_layout_dispatch (layout and dispatch in one call) against
the oracle: every layout output, the dispatch payload, scales, weights and
ids bit for bit, and the combine on the handle it returns.

In this call the dispatch loads and quantises the first source rows of each
CTA before the layout kernels are done.  The cases vary the token count,
source ranks that end inside a layout chunk, R from 1 to 64, K from 1 to 32,
empty and invalid slots, int32 indices, BF16 and both FP8 scale layouts,
both layout forms (one cluster kernel for small rank layouts, count + assign
otherwise), the expanded and fixed-capacity layouts, an empty batch and a
cached dispatch on the returned handle."""
import zlib

import numpy as np
import pytest
import torch

import ep_workloads as W
from tests import ep_harness as HN
from tests.test_parity_gpu import run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def _routing(T, K, E, seed, drop=0.0, bad=0.0):
    g = torch.Generator().manual_seed(seed)
    idx = torch.rand(T, E, generator=g).topk(min(K, E), dim=1).indices
    if drop > 0:
        idx = idx.masked_fill(torch.rand(T, K, generator=g) < drop, -1)
    if bad > 0:  # out-of-range values: flagged, treated as empty slots
        sel = torch.rand(T, K, generator=g) < bad
        idx = torch.where(sel, torch.full_like(idx, E + 3), idx)
    w = torch.rand(T, K, generator=g).masked_fill(idx < 0, 0.0)
    return idx.to(torch.int64).contiguous(), w.to(torch.float32).contiguous()


CASES = {
    # name: (T, K, E, R, H, M, fp8, col_major, drop, bad)
    "decode_like_fp8": (1024, 8, 256, 8, 1024, 128, True, False, 0.0, 0.0),
    "ragged_fp8_cm": (1000, 8, 64, 8, 512, 125, True, True, 0.05, 0.0),
    "bf16_src_inside_blocks": (777, 6, 48, 16, 256, 50, False, False, 0.1, 0.0),
    "r32_k4": (700, 4, 64, 32, 256, 22, True, False, 0.0, 0.0),
    "r1_k1": (300, 1, 5, 1, 128, 300, True, False, 0.1, 0.0),
    "k9_two_batches": (513, 9, 36, 4, 256, 129, True, True, 0.0, 0.0),
    "k32_four_batches": (512, 32, 64, 8, 128, 64, False, False, 0.05, 0.0),
    "invalid_indices": (257, 8, 32, 4, 256, 65, True, False, 0.05, 0.02),
    "one_token": (1, 8, 16, 4, 128, 1, True, False, 0.0, 0.0),
    "t_times_k_16384": (2048, 8, 64, 8, 128, 256, False, False, 0.0, 0.0),
}
# The cases on the count + assign kernels; the others take the cluster kernel.
TWO_KERNEL_CASES = {"bf16_src_inside_blocks", "r32_k4", "rank_t_times_k_above_16384", "rank_r64",
                    "expand_aligned", "fixed_capacity"}


@pytest.mark.parametrize("case", sorted(CASES))
def test_layout_dispatch_rank_layout(ep, case):
    T, K, E, R, H, M, fp8, cm, drop, bad = CASES[case]
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop, bad=bad)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 1, False, False, False, fp8, cm)
    r = run_and_check(ep, cfg, idx, x, w, bias0=True, fused=True)
    assert r["layout_kernels"] == (2 if case in TWO_KERNEL_CASES else 1)
    assert r["combine_mismatch"] == 0
    if bad > 0:
        assert r["lay"]["error"] & ep.EP_ERRBIT_BAD_TOPK_IDX


def test_layout_dispatch_int32_indices_and_no_weights(ep):
    T, K, E, R, H, M = 600, 8, 64, 8, 256, 75
    idx, w = _routing(T, K, E, seed=21, drop=0.05)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 1, False, False, False, True, False)
    r = run_and_check(ep, cfg, idx.to(torch.int32), x, w, bias0=False, fused=True)
    assert r["combine_mismatch"] == 0
    r = run_and_check(ep, cfg, idx, x, None, fused=True)   # no weights in, none out
    assert r["combine_mismatch"] == 0


EXPANDED_AND_WIDE = {
    # name: (T, K, E, R, H, M, A, expand, zero_pad, fp8, col_major, fixed)
    "rank_t_times_k_above_16384": (4096, 8, 256, 8, 256, 512, 1, False, False, True, False, False),
    "rank_r64": (1000, 4, 128, 64, 128, 16, 1, False, False, True, False, False),
    "expand_aligned": (600, 6, 32, 4, 256, 150, 16, True, True, True, True, False),
    "fixed_capacity": (512, 8, 64, 8, 256, 64, 1, True, False, True, True, True),
}


@pytest.mark.parametrize("case", sorted(EXPANDED_AND_WIDE))
def test_layout_dispatch_expanded_and_wide(ep, case):
    T, K, E, R, H, M, A, ex, zp, fp8, cm, fixed = EXPANDED_AND_WIDE[case]
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=0.05)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, A, ex, zp, False, fp8, cm, fixed_capacity=fixed)
    r = run_and_check(ep, cfg, idx, x, w, bias0=True, fused=True)
    assert r["layout_kernels"] == (2 if case in TWO_KERNEL_CASES else 1)
    assert r["combine_mismatch"] == 0


def test_layout_dispatch_back_to_back_calls(ep):
    """Consecutive calls whose handles reuse one another's device memory (the
    dispatch counters and control words a previous call left are reset by
    each layout): every output against the oracle, FP8 and BF16."""
    T, K, E, R, H, M = 1024, 8, 256, 8, 256, 128
    for i in range(8):
        fp8 = i % 2 == 0
        cfg = ep.make_config(T, K, E, R, H, M, 1, False, False, False, fp8, False)
        idx, w = _routing(T, K, E, seed=100 + i, drop=0.02)
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(200 + i)).to(torch.bfloat16)
        r = run_and_check(ep, cfg, idx, x, w, fused=True)
        assert r["layout_kernels"] == 1
        assert r["combine_mismatch"] == 0
        assert r["lay"]["error"] == 0


def test_layout_dispatch_empty(ep):
    cfg = ep.make_config(0, 4, 16, 4, 256, 8, 1, False, False, False, True, False)
    out = ep.alloc_recv_planned(cfg, with_weights=True, with_idx=True)
    idx = torch.empty((0, 4), dtype=torch.int64, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    h = ep.ep_layout_dispatch(cfg, idx, x, w, **out)
    g = HN.gpu_layout_arrays(h)
    assert g["totals"].tolist() == [0, 0] and int(g["error_word"][0]) == 0
    h.free()


def test_layout_dispatch_handle_reuse(ep):
    """A cached ep_dispatch on the handle of an ep_layout_dispatch call gives
    what ep_layout + ep_dispatch give (the call leaves the handle's dispatch
    counters reset)."""
    wl = W.WORKLOADS["decode"]
    T, H = 512, 1024
    cfg = ep.make_config(T, wl.num_topk, wl.num_experts, wl.num_ranks, H, 64, 1, False, False,
                         False, True, False)
    idx, w = _routing(T, wl.num_topk, wl.num_experts, seed=31)
    g = torch.Generator().manual_seed(8)
    x1 = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    x2 = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    out1 = ep.alloc_recv_planned(cfg, with_weights=True, with_idx=True)
    h = ep.ep_layout_dispatch(cfg, idx.cuda(), x1, w.cuda(), **out1)
    assert int(h.info.layout_kernels) in (1, 2)
    # zero-filled: rows past the real total are not written by either dispatch
    out2 = ep.alloc_recv(h, with_weights=True, with_idx=True, zero=True)
    ep.ep_dispatch(h, x2, w.cuda(), **out2)          # cached dispatch, new x
    ref = ep.ep_layout(cfg, idx.cuda())
    out3 = ep.alloc_recv(ref, with_weights=True, with_idx=True, zero=True)
    ep.ep_dispatch(ref, x2, w.cuda(), **out3)
    torch.cuda.synchronize()
    for k in out2:
        if out2[k] is not None:
            assert torch.equal(out2[k], out3[k]), k
    for n in ("dst_buffer_slot_idx", "recv_src_metadata", "psum_rank_src", "is_token_in_rank",
              "cnt_expert", "psum_expert", "totals", "error_word"):
        a, b = h.tensor(n), ref.tensor(n)
        if n == "recv_src_metadata":
            rows = int(ref.tensor("totals")[0])
            a, b = a[:rows], b[:rows]
        assert torch.equal(a, b), n
    h.free()
    ref.free()
