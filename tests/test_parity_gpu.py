"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Layout, metadata and dispatch payload (BF16 bytes, FP8 bytes and scales) must
match bit for bit; combine within 1 BF16 ulp per element (the kernel rounds
every operation exactly like the oracle, so in practice it is bit-exact and
the test also reports the number of differing elements).
"""
import zlib

import numpy as np
import pytest
import torch

import ep_workloads as W
from oracle import ep_oracle as O
from tests import ep_harness as HN

pytestmark = pytest.mark.gpu

COMBINE_ULP = 1  # tolerance stated for combine (1 BF16 ulp per element)


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def make_y(rows: int, H: int, seed: int, device) -> torch.Tensor:
    out = torch.empty((rows, H), dtype=torch.bfloat16, device=device)
    step = 8192
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = W.hashed_bf16_rows(torch.arange(r0, r1, device=device), H, seed, device)
    return out


def run_and_check(ep, cfg, idx_cpu, x_cpu, w_cpu, *, y_seed=11, combine_tokens=None,
                  dispatch_tokens=None, with_weights=True, with_idx=True, combine_w=True,
                  bias0=False, bias1=False, expert_bias=None, fused=False):
    """Layout, dispatch and combine through the C ABI against the oracle.
    fused: layout and dispatch by one ep_layout_dispatch call (no count
    wait), into buffers sized by ep_plan_layout."""
    dev = torch.device("cuda")
    idx = idx_cpu.to(dev)
    x = x_cpu.to(dev)
    w = w_cpu.to(dev) if w_cpu is not None else None
    lay = HN.oracle_layout(cfg, idx_cpu.to(torch.int64).numpy())
    use_fp8, cm = bool(cfg.use_fp8), bool(cfg.use_tma_aligned_col_major_sf)
    want_w, want_idx = with_weights and w is not None, with_idx and not cfg.do_expand
    if fused:
        out = ep.alloc_recv_planned(cfg, with_weights=want_w, with_idx=want_idx)
        h = ep.ep_layout_dispatch(cfg, idx, x, w, **out)
        HN.check_layout(h, lay)
    else:
        h = ep.ep_layout(cfg, idx)
        HN.check_layout(h, lay)
        out = ep.alloc_recv(h, with_weights=want_w, with_idx=want_idx)
        ep.ep_dispatch(h, x, w, **out)
    x_bits = HN.bits16(x_cpu)
    w_np = None if w_cpu is None else w_cpu.numpy()
    if dispatch_tokens is None:
        d_or = O.dispatch(lay, x_bits, w_np, use_fp8, cm, bool(cfg.do_zero_padding))
        HN.check_dispatch(h, lay, d_or, out, use_fp8, cm)
    else:
        d_or = HN.oracle_dispatch_tokens(x_bits, dispatch_tokens, use_fp8)
        HN.check_dispatch(h, lay, d_or, out, use_fp8, cm, tokens=dispatch_tokens)
        if cfg.do_expand and cfg.do_zero_padding:
            HN.check_padding_zero(lay, out, use_fp8, cm)

    # combine on a counter-based y so the oracle can rebuild any rows it needs
    T, H = cfg.num_tokens, cfg.hidden
    rows = h.rows_alloc
    y = make_y(rows, H, y_seed, dev)
    b0 = W.hashed_bf16_rows(torch.arange(T), H, y_seed + 1, dev) if bias0 else None
    b1 = W.hashed_bf16_rows(torch.arange(T), H, y_seed + 2, dev) if bias1 else None
    eb = expert_bias.to(dev) if expert_bias is not None else None
    cw = w if combine_w else None
    res = ep.ep_combine(h, y, cw, b0, b1, eb)
    torch.cuda.synchronize()
    toks = np.arange(T) if combine_tokens is None else np.asarray(combine_tokens)
    need = np.unique(lay["dst_buffer_slot_idx"][toks])
    need = need[need >= 0]
    y_bits = np.zeros((max(rows, 1), H), dtype=np.uint16)
    if need.size:
        y_bits[need] = HN.bits16(W.hashed_bf16_rows(torch.from_numpy(need), H, y_seed))
    ref = O.combine(lay, y_bits, None if cw is None else w_np,
                    None if b0 is None else HN.bits16(b0.cpu()),
                    None if b1 is None else HN.bits16(b1.cpu()),
                    None if eb is None else HN.bits16(expert_bias), tokens=toks)
    got = HN.bits16(res.index_select(0, torch.from_numpy(toks).to(dev)) if combine_tokens is not None
                    else res)
    d = HN.ulp_diff(got, ref)
    assert d.max(initial=0) <= COMBINE_ULP, f"combine max ulp diff {d.max(initial=0)}"
    kernels = int(h.info.layout_kernels)
    h.free()
    return {"lay": lay, "combine_mismatch": int((d != 0).sum()), "layout_kernels": kernels}


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed"])
def test_workload_parity(ep, name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl, seed=0)
    cfg = HN.cfg_for(ep, wl)
    T = wl.num_tokens
    big = T * wl.hidden > 4_000_000
    rng = np.random.default_rng(1)
    ct = np.sort(rng.choice(T, size=min(T, 384), replace=False)) if big else None
    r = run_and_check(ep, cfg, inp["topk_idx"], inp["x"], inp["topk_weights"],
                      combine_tokens=ct, bias0=(name == "tiny"), bias1=(name == "tiny"),
                      expert_bias=inp["expert_bias"])
    assert r["combine_mismatch"] == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed", "large"])
def test_workload_parity_reduced_tokens(ep, name):
    """Every workload's routing regime at a token count the oracle finishes fast,
    spanning several layout CTAs and a ragged last chunk; full combine parity."""
    wl = W.WORKLOADS[name]
    T = min(wl.num_tokens, 700)
    inp = W.make_inputs(wl, seed=5, num_tokens=T)
    cfg = HN.cfg_for(ep, wl, T=T, M=max(37, -(-T // wl.num_ranks)))
    run_and_check(ep, cfg, inp["topk_idx"], inp["x"], inp["topk_weights"],
                  expert_bias=inp["expert_bias"])


def test_large_full_size_sampled(ep):
    wl = W.WORKLOADS["large"]
    inp = W.make_inputs(wl, seed=0)
    cfg = HN.cfg_for(ep, wl)
    rng = np.random.default_rng(2)
    toks = np.sort(rng.choice(wl.num_tokens, size=256, replace=False))
    run_and_check(ep, cfg, inp["topk_idx"], inp["x"], inp["topk_weights"],
                  combine_tokens=toks, dispatch_tokens=toks)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------
def _routing(T, K, E, seed, drop=0.0, dup=False):
    g = torch.Generator().manual_seed(seed)
    if dup:
        idx = torch.randint(0, E, (T, K), generator=g)
    else:
        idx = torch.rand(T, E, generator=g).topk(min(K, E), dim=1).indices
        if K > E:
            idx = torch.cat([idx, torch.full((T, K - E), -1, dtype=idx.dtype)], 1)
    if drop > 0:
        idx = idx.masked_fill(torch.rand(T, K, generator=g) < drop, -1)
    w = torch.rand(T, K, generator=g).masked_fill(idx < 0, 0.0)
    return idx.to(torch.int64).contiguous(), w.to(torch.float32).contiguous()


EDGE = {
    # name: (T, K, E, R, H, M, A, expand, zero_pad, sync, fp8, col_major, drop, dup)
    "empty_tokens": (0, 4, 8, 2, 256, 4, 4, True, True, True, True, True, 0.0, False),
    "empty_tokens_rank": (0, 4, 8, 2, 64, 4, 1, False, False, False, False, False, 0.0, False),
    "all_slots_empty": (50, 3, 8, 4, 128, 13, 4, True, True, True, True, False, 1.0, False),
    "all_empty_nosync": (50, 3, 8, 4, 64, 13, 4, True, True, False, False, False, 1.0, False),
    "one_token": (1, 2, 4, 2, 128, 1, 8, True, True, True, True, True, 0.0, False),
    "k1_r1": (300, 1, 5, 1, 72, 300, 1, True, False, True, False, False, 0.1, False),
    "l1_rank_layout": (257, 6, 8, 8, 128, 33, 1, False, False, True, True, False, 0.2, False),
    "ragged_bf16_h": (333, 4, 16, 4, 8 * 37, 100, 3, True, True, True, False, False, 0.1, False),
    "ragged_fp8_h": (333, 4, 16, 4, 128 * 3, 100, 16, True, True, True, True, True, 0.1, False),
    "fp8_rowmajor_expand": (200, 8, 32, 4, 512, 64, 32, True, True, True, True, False, 0.0, False),
    "big_alignment": (90, 2, 8, 2, 128, 45, 256, True, True, True, True, True, 0.0, False),
    "no_zero_padding": (128, 4, 16, 4, 256, 32, 8, True, False, True, True, True, 0.05, False),
    "rank_nosync_fp8": (512, 8, 64, 8, 1024, 64, 1, False, False, False, True, False, 0.0, False),
    "expand_nosync": (512, 8, 64, 8, 256, 64, 16, True, True, False, False, False, 0.0, False),
    "dup_experts_sync_expand": (100, 6, 8, 2, 128, 50, 4, True, True, True, True, True, 0.1, True),
    "dup_experts_rank": (100, 6, 8, 2, 128, 50, 1, False, False, True, False, False, 0.1, True),
    "many_src_ranks_small_m": (1000, 4, 32, 32, 64, 32, 2, True, True, True, False, False, 0.0, False),
    "max_topk": (64, 32, 64, 4, 128, 16, 4, True, True, True, True, True, 0.0, False),
    "many_experts": (256, 8, 2048, 16, 128, 16, 4, True, True, True, True, True, 0.0, False),
    # Rank layouts of up to 15 chunks run as one thread-block cluster (a CTA
    # per chunk and one more), larger ones and the expanded layouts as two
    # kernels: both sides of the boundary, and three ragged chunks per source
    # rank.
    "chunks_15_rank_sync": (960, 5, 48, 16, 256, 64, 1, False, False, True, True, False, 0.05,
                            False),
    "chunks_16_rank_nosync": (1024, 4, 32, 16, 128, 64, 1, False, False, False, True, False,
                              0.05, False),
    "chunks_16_expand_sync": (1000, 6, 64, 16, 256, 63, 8, True, True, True, True, True, 0.05,
                              False),
    "chunks_17_expand_sync": (1020, 6, 34, 17, 256, 60, 8, True, True, True, True, True, 0.05,
                              False),
    "chunks_17_rank_nosync": (1020, 4, 34, 17, 128, 60, 1, False, False, False, False, False,
                              0.0, False),
    "chunks_9_three_per_source": (1500, 8, 24, 3, 256, 700, 4, True, True, True, True, False,
                                  0.1, True),
    # Few slots and a long row: the combine's chunk is 16 KB (top-1 with a
    # per-token bias), so each of 224 consumer threads reduces pairs of 16-byte
    # vectors three times over and the last pass is ragged (1024 vectors).
    "k1_wide_row_many_vectors": (300, 1, 8, 4, 16384, 75, 1, False, False, True, False, False,
                                 0.05, False),
    "k2_wide_row_expand": (200, 2, 8, 4, 16384, 50, 4, True, True, False, True, False, 0.05,
                           False),
}


# Layout form the boundary cases must take: 1 = the cluster kernel, 2 = the
# count and assign kernels.
EDGE_FORM = {
    "chunks_15_rank_sync": 1,
    "chunks_16_rank_nosync": 2,
    "chunks_16_expand_sync": 2,
    "chunks_17_expand_sync": 2,
    "chunks_17_rank_nosync": 2,
    "chunks_9_three_per_source": 2,
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases(ep, case):
    T, K, E, R, H, M, A, ex, zp, sync, fp8, cm, drop, dup = EDGE[case]
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop, dup=dup)
    g = torch.Generator().manual_seed(3)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, A, ex, zp, sync, fp8, cm)
    r = run_and_check(ep, cfg, idx, x, w, bias0=True)
    if case in EDGE_FORM:
        assert r["layout_kernels"] == EDGE_FORM[case]


def test_combine_variants(ep):
    """No weights (rows used once), per-token biases, per-expert bias, both layouts."""
    T, K, E, R, H, M = 300, 6, 16, 4, 256, 75
    idx, w = _routing(T, K, E, seed=4, drop=0.1, dup=True)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    eb = W.hashed_bf16_rows(torch.arange(E), H, 99)
    for expand in (False, True):
        for combine_w in (True, False):
            for b0, b1, e_b in [(False, False, None), (True, False, None), (False, True, eb),
                                (True, True, eb)]:
                run_and_check(ep, ep.make_config(T, K, E, R, H, M, 4 if expand else 1, expand,
                                                 expand, True),
                              idx, x, w, combine_w=combine_w, bias0=b0, bias1=b1, expert_bias=e_b)


def test_int32_topk_idx(ep):
    T, K, E, R, H, M = 400, 4, 32, 8, 128, 50
    idx, w = _routing(T, K, E, seed=8, drop=0.1)
    x = torch.randn(T, H).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 8, True, True, True, True, True)
    run_and_check(ep, cfg, idx.to(torch.int32), x, w)


def test_fp8_special_values(ep):
    T, K, E, R, H = 16, 2, 4, 2, 512
    idx = torch.tensor([[0, 3]] * T, dtype=torch.int64)
    w = torch.full((T, K), 0.5)
    xf = torch.randn(T, H, generator=torch.Generator().manual_seed(1))
    xf[0, :128] = 0.0                    # zero block -> scale 0, zero bytes
    xf[1, :] = -0.0                      # negative zeros
    xf[2, :128] *= 1e-38                 # subnormal BF16 inputs, subnormal scale
    xf[3, :] = 1.0                       # constant blocks
    xf[4, :] = torch.tensor(np.random.default_rng(0).standard_cauchy(H), dtype=torch.float32)
    xf[5, 5] = 3.0e38                    # near the BF16 maximum
    xf[6, :] = torch.linspace(-448, 448, H)
    xf[7, 0:128:2] = 1e-30
    cfg = ep.make_config(T, K, E, R, H, 8, 4, True, True, True, True, True)
    run_and_check(ep, cfg, idx, xf.to(torch.bfloat16), w)


@pytest.mark.parametrize("col_major", [False, True])
def test_fp8_non_finite_inputs(ep, col_major):
    """NaN and +-Inf activations (reading R16): a block holding a NaN gets a
    NaN scale and 0x7F in every byte; a block whose amax is infinite gets
    scale +inf, signed zeros for its finite elements and 0x7F for its
    infinite ones.  Bytes compared exactly with the oracle, scales with NaN
    equal to NaN; the other blocks are unaffected."""
    T, K, E, R, H = 12, 2, 4, 2, 512
    idx = torch.tensor([[0, 3]] * T, dtype=torch.int64)
    w = torch.full((T, K), 0.5)
    xf = torch.randn(T, H, generator=torch.Generator().manual_seed(2))
    xf[0, 5] = float("nan")
    xf[1, 130] = -float("nan")
    xf[1, 131] = float("inf")
    xf[2, 260] = float("inf")
    xf[3, 400] = -float("inf")
    xf[3, 401] = float("inf")
    xf[4, :128] = float("inf")
    xf[5, 256:384] = float("nan")
    xf[6, :] = -float("inf")
    xf[7, 0] = float("nan")
    xf[7, 128] = float("inf")
    xf[7, 256] = -float("inf")
    cfg = ep.make_config(T, K, E, R, H, 8, 4, True, True, True, True, col_major)
    dev = torch.device("cuda")
    h = ep.ep_layout(cfg, idx.to(dev))
    lay = HN.oracle_layout(cfg, idx.numpy())
    HN.check_layout(h, lay)
    out = ep.alloc_recv(h, with_weights=True)
    x = xf.to(torch.bfloat16)
    ep.ep_dispatch(h, x.to(dev), w.to(dev), **out)
    d_or = O.dispatch(lay, HN.bits16(x), w.numpy(), True, col_major, True)
    HN.check_dispatch(h, lay, d_or, out, True, col_major)
    q, s = O.quantize_row(HN.bits16(x))
    assert np.isnan(s[0, 0]) and np.all(q[0, :128] == 0x7F)
    assert s[4, 0] == np.inf and np.all(q[4, :128] == 0x7F)
    h.free()


def test_bad_topk_idx_values(ep):
    T, K, E, R, H, M = 40, 3, 8, 2, 128, 20
    idx, w = _routing(T, K, E, seed=12)
    idx[0, 1] = 8
    idx[5, 0] = -7
    idx[9, 2] = 1 << 40
    x = torch.randn(T, H).to(torch.bfloat16)
    for sync in (True, False):
        cfg = ep.make_config(T, K, E, R, H, M, 4, True, True, sync, False)
        h = ep.ep_layout(cfg, idx.cuda())
        if sync:
            assert h.status == ep.EP_ERR_BAD_TOPK_IDX
        lay = HN.oracle_layout(cfg, idx.numpy())
        assert lay["error"] == 1
        HN.check_layout(h, lay)
        h.free()
        run_and_check(ep, cfg, idx, x, w)


def test_overflow_with_repeated_experts(ep):
    """No-sync expanded layout whose routing repeats experts beyond the printed
    per-rank bound: rows past the allocation are dropped and flagged, and no
    kernel writes past the caller's buffers (canary rows stay intact)."""
    T, K, E, R, H, M = 2, 4, 2, 2, 128, 1
    idx = torch.tensor([[0, 0, 0, 0], [1, 1, 0, 0]], dtype=torch.int64)
    w = torch.full((T, K), 0.25)
    x = torch.randn(T, H).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 1, True, True, False, True, True)
    h = ep.ep_layout(cfg, idx.cuda())
    lay = HN.oracle_layout(cfg, idx.numpy())
    assert lay["error"] & 2 and h.rows_alloc == 4
    HN.check_layout(h, lay)
    canary = 5
    big = torch.full((h.rows_alloc + canary, H), 0xA5, dtype=torch.uint8, device="cuda")
    sf = torch.full((int(h.info.sf_numel) + 64,), -7.0, device="cuda")
    rw = torch.full((h.rows_alloc + canary,), -3.0, device="cuda")
    ep.ep_dispatch(h, x.cuda(), w.cuda(), big[:h.rows_alloc], sf[:int(h.info.sf_numel)],
                   rw[:h.rows_alloc])
    torch.cuda.synchronize()
    assert int((big[h.rows_alloc:] != 0xA5).sum()) == 0
    assert int((sf[int(h.info.sf_numel):] != -7.0).sum()) == 0
    assert int((rw[h.rows_alloc:] != -3.0).sum()) == 0
    h.free()
    run_and_check(ep, cfg, idx, x, w)


def test_output_canaries(ep):
    """Dispatch and combine write nothing outside the rows they own."""
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, seed=3)
    cfg = HN.cfg_for(ep, wl)
    h = ep.ep_layout(cfg, inp["topk_idx"].cuda())
    rows, H, T = h.rows_alloc, wl.hidden, wl.num_tokens
    pad = 7
    rx = torch.full(((rows + pad) * H,), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rw = torch.full((rows + pad,), 123.0, device="cuda")
    ep.ep_dispatch(h, inp["x"].cuda(), inp["topk_weights"].cuda(),
                   rx[:rows * H].view(rows, H), None, rw[:rows])
    out = torch.full(((T + pad) * H,), 0x3C3C, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    y = make_y(rows, H, 3, "cuda")
    ep.ep_combine(h, y, inp["topk_weights"].cuda(), out=out[:T * H].view(T, H))
    torch.cuda.synchronize()
    assert int((rx.view(torch.int16)[rows * H:] != 0x5A5A).sum()) == 0
    assert int((rw[rows:] != 123.0).sum()) == 0
    assert int((out.view(torch.int16)[T * H:] != 0x3C3C).sum()) == 0
    h.free()


def test_num_sms_cap_same_result(ep):
    wl = W.WORKLOADS["prefill"]
    inp = W.make_inputs(wl, seed=9, num_tokens=512)
    for sms in (1, 3, 0):
        cfg = HN.cfg_for(ep, wl, T=512, M=64, num_sms=sms)
        run_and_check(ep, cfg, inp["topk_idx"], inp["x"], inp["topk_weights"])


def test_layout_deterministic_and_cached_dispatch(ep):
    """Two layouts of the same routing agree; one handle serves a second x."""
    wl = W.WORKLOADS["skewed"]
    T = 3000
    inp = W.make_inputs(wl, seed=4, num_tokens=T)
    cfg = HN.cfg_for(ep, wl, T=T, M=400)
    idx = inp["topk_idx"].cuda()
    h1, h2 = ep.ep_layout(cfg, idx), ep.ep_layout(cfg, idx)
    a, b = HN.gpu_layout_arrays(h1), HN.gpu_layout_arrays(h2)
    total = int(a["totals"][0])                 # rank layout: rows past it are unspecified
    a["recv_src_metadata"] = a["recv_src_metadata"][:total]
    b["recv_src_metadata"] = b["recv_src_metadata"][:total]
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    lay = HN.oracle_layout(cfg, inp["topk_idx"].numpy())
    for seed in (1, 2):
        x = W.make_x(wl, seed, num_tokens=T)
        out = ep.alloc_recv(h1)
        ep.ep_dispatch(h1, x.cuda(), None, **out)
        d_or = O.dispatch(lay, HN.bits16(x), None, False, False, False)
        HN.check_dispatch(h1, lay, d_or, out, False, False)
    h1.free()
    h2.free()


@pytest.mark.parametrize("name,T", [("decode", None), ("large", 2048)])
@pytest.mark.parametrize("one_call", [False, True])
def test_cuda_graph_capture_and_replay(ep, name, T, one_call):
    """Without the host count wait the whole path is stream-ordered: capture
    layout + dispatch + combine (+ handle free) in a CUDA graph, replay it on
    new inputs copied into the captured buffers, and compare with an eager
    run of the same inputs.  one_call: layout and dispatch captured as one
    ep_layout_dispatch call (its early source-row loads ride on the
    programmatic-dependent-launch edge of the graph)."""
    wl = W.WORKLOADS[name]
    T = wl.num_tokens if T is None else T
    cfg = HN.cfg_for(ep, wl, T=T, do_cpu_sync=False)
    K, H = wl.num_topk, wl.hidden
    rows = ep.upper_bound_rows(cfg)
    dev = torch.device("cuda")
    idx_s = torch.empty((T, K), dtype=torch.int64, device=dev)
    w_s = torch.empty((T, K), dtype=torch.float32, device=dev)
    x_s = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    y_s = make_y(rows, H, 21, dev)
    nb = H // 128
    sfn = O.sf_numel(rows, H, wl.col_major_sf) if wl.use_fp8 else 0
    recv = {"recv_x": torch.zeros((rows, H), dtype=torch.uint8 if wl.use_fp8 else torch.bfloat16,
                                  device=dev),
            "recv_sf": torch.zeros((sfn,), dtype=torch.float32, device=dev) if wl.use_fp8 else None,
            "recv_topk_weights": torch.zeros((rows,) if wl.do_expand else (rows, K),
                                             dtype=torch.float32, device=dev)}
    res = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def fill(seed):
        inp = W.make_inputs(wl, seed, num_tokens=T)
        idx_s.copy_(inp["topk_idx"])
        w_s.copy_(inp["topk_weights"])
        x_s.copy_(inp["x"])

    def path(st):
        if one_call:
            h = ep.ep_layout_dispatch(cfg, idx_s, x_s, w_s, stream=st, **recv)
        else:
            h = ep.ep_layout(cfg, idx_s, stream=st)
            ep.ep_dispatch(h, x_s, w_s, stream=st, **recv)
        ep.ep_combine(h, y_s, w_s, out=res, stream=st)
        h.free()

    s = torch.cuda.Stream()
    fill(0)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        path(s)                           # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        path(s)
    for seed in (7, 8):
        fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in recv.items() if v is not None}
        got_res = res.clone()
        h = ep.ep_layout(cfg, idx_s)
        total = int(h.tensor("totals").cpu()[1 if wl.do_expand else 0])
        eager = ep.alloc_recv(h, with_weights=True)
        ep.ep_dispatch(h, x_s, w_s, **eager)
        ref = ep.ep_combine(h, y_s, w_s)
        torch.cuda.synchronize()
        assert torch.equal(got["recv_x"][:total], eager["recv_x"][:total])
        if wl.use_fp8:
            if wl.col_major_sf:
                st = -(-rows // 4) * 4
                a = got["recv_sf"].view(nb, st)[:, :total]
                b = eager["recv_sf"].view(nb, st)[:, :total]
            else:
                a = got["recv_sf"].view(rows, nb)[:total]
                b = eager["recv_sf"].view(rows, nb)[:total]
            assert torch.equal(a, b)
        assert torch.equal(got["recv_topk_weights"][:total], eager["recv_topk_weights"][:total])
        assert torch.equal(got_res, ref)
        h.free()


def test_shared_memory_window_edges(ep):
    """Shapes whose dynamic shared memory is exactly the 48 KB default window
    (which the kernels' static shared memory pushes past): the combine with a
    per-expert bias at hidden 7168 and top-8, and the BF16 dispatch at hidden
    8192."""
    T, K, E, R, H, M = 64, 8, 16, 4, 7168, 16
    idx, w = _routing(T, K, E, seed=21)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    eb = W.hashed_bf16_rows(torch.arange(E), H, 17)
    run_and_check(ep, ep.make_config(T, K, E, R, H, M, 4, True, True, True),
                  idx, x, w, expert_bias=eb)
    T, K, E, R, H, M = 48, 2, 8, 2, 8192, 24
    idx, w = _routing(T, K, E, seed=22)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    run_and_check(ep, ep.make_config(T, K, E, R, H, M, 1, False, False, True), idx, x, w)


@pytest.mark.parametrize("fp8,cm", [(True, True), (True, False), (False, False)])
def test_maximum_hidden(ep, fp8, cm):
    """The largest hidden size the configuration accepts (32768): a quantising
    dispatch needs more shared memory per stage than three stages leave room
    for, so its stage ring is shorter; every output still matches the oracle
    (with a per-expert bias in the combine)."""
    T, K, E, R, H, M = 40, 4, 8, 2, 32768, 20
    idx, w = _routing(T, K, E, seed=23, drop=0.1)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    eb = W.hashed_bf16_rows(torch.arange(E), H, 19)
    run_and_check(ep, ep.make_config(T, K, E, R, H, M, 8, True, True, True, fp8, cm),
                  idx, x, w, expert_bias=eb)


@pytest.mark.parametrize("cm_in", [False, True])
def test_maximum_hidden_prequantised(ep, cm_in):
    from tests.test_prequant_gpu import run_prequant
    T, K, E, R, H, M = 40, 4, 8, 2, 32768, 20
    idx, w = _routing(T, K, E, seed=24, drop=0.1)
    run_prequant(ep, ep.make_config(T, K, E, R, H, M, 8, True, True, False, True, True),
                 idx, w, cm_in)


def test_maximum_hidden_backward_pair(ep):
    from tests.test_backward_gpu import check_backward
    T, K, E, R, H, M = 40, 4, 8, 2, 32768, 20
    idx, _ = _routing(T, K, E, seed=25, drop=0.1)
    check_backward(ep, ep.make_config(T, K, E, R, H, M, 8, True, True, False, False, False), idx)


def test_short_combine_grid_strides(ep):
    """Short combines (at most 16 units per CTA) step each CTA's (token,
    chunk) by the grid stride with adds only, also without a per-expert bias.
    Hidden 7168 splits into 4 chunks; grids of 2, 6 and 10 CTAs (1, 3 and 5
    SMs) over 7 to 37 tokens give strides that wrap a row end and up to 16
    units per CTA, and 64 tokens on the full grid one unit per CTA.
    Weighted with a per-token bias, and unweighted; both layouts; every
    output against the oracle."""
    K, E, R, H = 8, 32, 4, 7168
    for T, sms in ((7, 1), (23, 3), (37, 5), (64, 0)):
        M = (T + R - 1) // R
        idx, w = _routing(T, K, E, seed=40 + T, drop=0.05)
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
        for expand in (False, True):
            cfg = ep.make_config(T, K, E, R, H, M, 4 if expand else 1, expand, expand, True,
                                 num_sms=sms)
            run_and_check(ep, cfg, idx, x, w, bias0=True)
            run_and_check(ep, cfg, idx, x, w, combine_w=False)


@pytest.mark.parametrize("expand", [False, True])
def test_expert_bias_combine_grid_strides(ep, expand):
    """The per-expert-bias combine steps each CTA's (token, chunk) by the grid
    stride with adds only.  Hidden 7168 splits into 7 chunks (10 with a
    per-token bias); capping the grid at 1 and 3 SMs, and the full grid, gives
    strides of fewer chunks than a row, strides that wrap a row end, and
    several units per CTA.  Every output against the oracle."""
    T, K, E, R, H, M = 600, 8, 32, 4, 7168, 150
    idx, w = _routing(T, K, E, seed=26, drop=0.05)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    eb = W.hashed_bf16_rows(torch.arange(E), H, 27)
    for sms in (1, 3, 0):
        for b0 in (False, True):
            cfg = ep.make_config(T, K, E, R, H, M, 4 if expand else 1, expand, expand, True,
                                 num_sms=sms)
            run_and_check(ep, cfg, idx, x, w, bias0=b0, expert_bias=eb)
