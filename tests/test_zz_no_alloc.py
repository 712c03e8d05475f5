"""ep_layout_noalloc: the routing layout for callers that cannot allocate.

Code running inside a CUDA-graph capture that must not add allocation nodes,
or runtimes that own all device memory up front, cannot let the library call
cudaMalloc.  ep_layout_noalloc takes every output buffer from the caller and
keeps its scratch in a static device array.  These tests call it through the
C ABI and check that two calls in a row give exactly (bit for bit, the
tolerance every layout test uses) what ep_layout gives -- also for the
fixed-capacity layout, int32 indices, an empty batch and replays of a CUDA
graph that captured the call -- and that a problem too big for the static
scratch is refused before any GPU work.  ep_layout itself is compared with
the CPU oracle by the parity tests.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import ep_workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def _layout_via_handle(ep, cfg, idx):
    h = ep.ep_layout(cfg, idx)
    torch.cuda.synchronize()
    names = ["topk_idx", "cnt_expert", "cnt_expert_aligned", "psum_expert", "cnt_rank",
             "psum_rank", "psum_rank_src", "dst_buffer_slot_idx", "recv_src_metadata",
             "is_token_in_rank", "totals", "error_word"]
    out = {n: h.tensor(n).cpu().numpy() for n in names}
    h.free()
    return out


def _compare(ep, cfg, idx):
    ref = _layout_via_handle(ep, cfg, idx)
    buf = ep.alloc_layout_buffers(cfg)
    st = ep.ep_layout_noalloc(cfg, idx, buf)
    assert st == ep.EP_OK, ep.status_string(st)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in buf.items()}
    pairs = [("topk_idx32", "topk_idx"), ("cnt_expert", "cnt_expert"),
             ("cnt_expert_aligned", "cnt_expert_aligned"), ("psum_expert", "psum_expert"),
             ("cnt_rank", "cnt_rank"), ("psum_rank", "psum_rank"),
             ("psum_rank_src", "psum_rank_src"), ("dst_buffer_slot_idx", "dst_buffer_slot_idx"),
             ("is_token_in_rank", "is_token_in_rank")]
    for a, b in pairs:
        assert np.array_equal(got[a], ref[b]), a
    if cfg.fixed_capacity:
        # expert e's rows start at e * capacity; only the first count are written
        cap = cfg.num_max_tokens_per_rank * cfg.num_ranks
        cnt = np.minimum(ref["cnt_expert"], cap)
        used = np.concatenate([e * cap + np.arange(c) for e, c in enumerate(cnt)]).astype(np.int64)
        assert np.array_equal(got["recv_src_metadata"][used], ref["recv_src_metadata"][used])
    else:
        total = int(ref["totals"][1] if cfg.do_expand else ref["totals"][0])
        rows = min(total, got["recv_src_metadata"].shape[0])
        assert np.array_equal(got["recv_src_metadata"][:rows], ref["recv_src_metadata"][:rows])
    assert got["status"][2] == ref["totals"][0] and got["status"][3] == ref["totals"][1]
    assert int(got["status"][0]) == int(ref["error_word"][0])
    # padding prefix: aligned minus unaligned counts, summed
    pad = np.concatenate([[0], np.cumsum(got["cnt_expert_aligned"] - got["cnt_expert"])])
    assert np.array_equal(got["psum_padding"], pad)


def test_noalloc_two_calls_match_layout(ep):
    dev = torch.device("cuda")
    # first call: expanded layout with alignment padding (prefill routing)
    wl = W.WORKLOADS["prefill"]
    idx, _ = W.make_routing(wl, seed=0)
    cfg = ep.make_config(wl.num_tokens, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden,
                         wl.num_max_tokens_per_rank, wl.expert_alignment, True, True, False,
                         True, True)
    _compare(ep, cfg, idx.to(dev))
    # second call, right after: rank layout, other sizes (skewed routing), so
    # the scratch holds the first call's histograms when it starts
    wl = W.WORKLOADS["skewed"]
    idx, _ = W.make_routing(wl, seed=1, num_tokens=5000)
    cfg = ep.make_config(5000, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden, 700,
                         1, False, False, False, False, False)
    _compare(ep, cfg, idx.to(dev))


def test_noalloc_fixed_capacity_int32_and_empty(ep):
    """The fixed-capacity layout, int32 topk_idx, and a batch with no tokens."""
    dev = torch.device("cuda")
    wl = W.WORKLOADS["decode_ll"]
    idx, _ = W.make_routing(wl, seed=2)
    cfg = ep.make_config(wl.num_tokens, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden,
                         wl.num_max_tokens_per_rank, 1, True, False, False, True, True,
                         fixed_capacity=True)
    _compare(ep, cfg, idx.to(dev))
    wl = W.WORKLOADS["skewed"]
    idx, _ = W.make_routing(wl, seed=3, num_tokens=3000)
    cfg = ep.make_config(3000, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden, 400,
                         4, True, True, False, False, False)
    _compare(ep, cfg, idx.to(torch.int32).to(dev))
    cfg = ep.make_config(0, 4, 16, 4, 256, 8, 4, True, True, False)
    _compare(ep, cfg, torch.empty((0, 4), dtype=torch.int64, device=dev))


def test_noalloc_graph_capture_and_replay(ep):
    """Graph capture is the case that cannot allocate: one call outside the
    capture, then the call captured into a CUDA graph and replayed on new
    routing written into the captured input; each replay against
    ep_layout of the same routing."""
    dev = torch.device("cuda")
    wl = W.WORKLOADS["decode"]
    T, K = wl.num_tokens, wl.num_topk
    cfg = ep.make_config(T, K, wl.num_experts, wl.num_ranks, wl.hidden,
                         wl.num_max_tokens_per_rank, 1, False, False, False, True, False)
    idx_s = torch.empty((T, K), dtype=torch.int64, device=dev)
    buf = ep.alloc_layout_buffers(cfg)
    idx_s.copy_(W.make_routing(wl, seed=0)[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        assert ep.ep_layout_noalloc(cfg, idx_s, buf, stream=s) == ep.EP_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = ep.ep_layout_noalloc(cfg, idx_s, buf, stream=s)
    assert st == ep.EP_OK
    for seed in (5, 6):
        idx_s.copy_(W.make_routing(wl, seed=seed)[0])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in buf.items()}
        ref = _layout_via_handle(ep, cfg, idx_s)
        for a, b in [("topk_idx32", "topk_idx"), ("cnt_expert", "cnt_expert"),
                     ("psum_rank", "psum_rank"), ("psum_rank_src", "psum_rank_src"),
                     ("dst_buffer_slot_idx", "dst_buffer_slot_idx"),
                     ("is_token_in_rank", "is_token_in_rank")]:
            assert np.array_equal(got[a], ref[b]), a
        total = int(ref["totals"][0])
        assert np.array_equal(got["recv_src_metadata"][:total], ref["recv_src_metadata"][:total])
        assert got["status"][2] == total


def test_noalloc_refuses_oversized_and_sync(ep):
    dev = torch.device("cuda")
    dummy = torch.zeros(16, dtype=torch.int64, device=dev)
    buf = {n: dummy for n, _ in ep.EpLayoutBuffersC._fields_}
    # 2048 experts over 16 ranks: each 256-token chunk needs 2065 scratch words
    T = 256 * 300
    cfg = ep.make_config(T, 8, 2048, 16, 128, T // 16 + 1, 1, True, False, False)
    chunks = -(-T // cfg.num_max_tokens_per_rank) * -(-min(cfg.num_max_tokens_per_rank, T) // 256)
    assert chunks * (2048 + 16 + 1) > ep.EP_NOALLOC_SCRATCH_WORDS
    assert ep.ep_layout_noalloc(cfg, dummy, buf) == ep.EP_ERR_UNSUPPORTED
    cfg = ep.make_config(128, 2, 16, 4, 256, 32, 8, True, True, True)
    assert ep.ep_layout_noalloc(cfg, dummy, buf) == ep.EP_ERR_INVALID_ARG
