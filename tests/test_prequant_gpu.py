"""GPU parity of dispatch with a pre-quantised FP8 input ("DeepEP V2 notes,
ch. 7" §7.1: x may be an FP8 data + scale-factor tuple; §7.3: the scale
factors land row-major or TMA-aligned column-major) against the oracle.

Bytes, scales (bit patterns), weights and local expert ids must match
exactly; the input scales come row-major or as a column-major view.
"""
import zlib

import numpy as np
import pytest
import torch

import ep_workloads as W
from oracle import ep_oracle as O
from tests import ep_harness as HN

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


def make_scales(T, nb, seed, col_major_input, dev):
    """fp32 scales [T, nb]: row-major, or a column-major view with token
    stride 1 and block stride align(T, 4) (the TMA-aligned layout)."""
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(T, nb, generator=g).abs() * 0.01
    if T > 0:
        s[0, 0] = -0.0
    if not col_major_input:
        return s.to(dev).contiguous()
    st = -(-max(T, 1) // 4) * 4
    store = torch.full((nb, st), 99.0, device=dev)
    store[:, :T] = s.t().to(dev)
    return store[:, :T].t()


def run_prequant(ep, cfg, idx_cpu, w_cpu, col_major_input, seed=3, canary=4):
    dev = torch.device("cuda")
    T, H = cfg.num_tokens, cfg.hidden
    nb = H // 128
    h = ep.ep_layout(cfg, idx_cpu.to(dev))
    lay = HN.oracle_layout(cfg, idx_cpu.numpy())
    HN.check_layout(h, lay)
    g = torch.Generator().manual_seed(seed)
    xq = torch.randint(0, 256, (T, H), generator=g, dtype=torch.uint8)
    if T > 0:
        xq[0, :256 if H >= 256 else H] = torch.arange(256, dtype=torch.int32)[:min(H, 256)].to(torch.uint8)
    xs = make_scales(T, nb, seed + 1, col_major_input, dev)
    w = w_cpu.to(dev)
    rows = h.rows_alloc
    cm = bool(cfg.use_tma_aligned_col_major_sf)
    big_x = torch.full((rows + canary, H), 0xA5, dtype=torch.uint8, device=dev)
    sfn = int(h.info.sf_numel)
    big_sf = torch.full((sfn + canary,), -7.0, device=dev)
    shape_w = (rows + canary,) if cfg.do_expand else (rows + canary, cfg.num_topk)
    big_w = torch.full(shape_w, -3.0, device=dev)
    out = {"recv_x": big_x[:rows], "recv_sf": big_sf[:sfn], "recv_topk_weights": big_w[:rows],
           "recv_topk_idx": None if cfg.do_expand else
           torch.empty((rows, cfg.num_topk), dtype=torch.int32, device=dev)}
    ep.ep_dispatch_fp8(h, xq.to(dev), xs, w, **out)
    torch.cuda.synchronize()
    d_or = O.dispatch_prequantised(lay, xq.numpy(), xs.cpu().numpy(), w_cpu.numpy(), cm,
                                   bool(cfg.do_zero_padding))
    HN.check_dispatch(h, lay, d_or, out, True, cm)
    # scale bit patterns (the float compare above cannot tell -0 from 0)
    pdef = np.flatnonzero(d_or["payload_defined"][:rows])
    gs = out["recv_sf"].cpu().numpy().view(np.uint32)
    for j in range(nb):
        ix = O.sf_index(pdef, j, rows, H, cm, lay.get("capacity"))
        assert np.array_equal(gs[ix], d_or["recv_sf"][ix].view(np.uint32)), f"sf bits block {j}"
    assert bool((big_x[rows:] == 0xA5).all()), "payload written past rows_alloc"
    assert bool((big_sf[sfn:] == -7.0).all()), "scales written past sf_numel"
    assert bool((big_w[rows:] == -3.0).all()), "weights written past rows_alloc"
    if cfg.do_expand and cfg.do_zero_padding:
        HN.check_padding_zero(lay, out, True, cm)
    h.free()


CASES = {
    # name: (T, K, E, R, H, M, A, expand, zero_pad, sync, col_major_out, col_major_in, drop, dup)
    "expand_cm_from_rowmajor": (700, 8, 64, 8, 512, 100, 16, True, True, True, True, False, 0.1, False),
    "expand_cm_from_colmajor": (700, 8, 64, 8, 512, 100, 16, True, True, True, True, True, 0.1, False),
    "expand_rm_from_colmajor": (333, 4, 16, 4, 384, 100, 8, True, True, True, False, True, 0.1, False),
    "expand_rm_from_rowmajor": (333, 4, 16, 4, 384, 100, 8, True, True, True, False, False, 0.1, False),
    "expand_no_zero_pad": (300, 4, 16, 4, 256, 75, 8, True, False, True, True, False, 0.0, False),
    "rank_rm": (513, 8, 64, 8, 1024, 65, 1, False, False, True, False, False, 0.1, False),
    "rank_cm_nosync": (600, 8, 32, 8, 256, 75, 1, False, False, False, True, True, 0.0, False),
    "expand_nosync_odd_blocks": (500, 6, 32, 4, 128 * 5, 125, 4, True, True, False, True, False, 0.0, False),
    "dup_experts_expand": (100, 6, 8, 2, 128, 50, 4, True, True, True, True, False, 0.1, True),
    "dup_experts_rank": (100, 6, 8, 2, 128, 50, 1, False, False, True, False, True, 0.1, True),
    "empty_tokens": (0, 4, 8, 2, 256, 4, 4, True, True, True, True, False, 0.0, False),
    "all_slots_empty": (50, 3, 8, 4, 128, 13, 4, True, True, True, False, False, 1.0, False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prequantised_dispatch(ep, case):
    T, K, E, R, H, M, A, ex, zp, sync, cmo, cmi, drop, dup = CASES[case]
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop, dup=dup)
    cfg = ep.make_config(T, K, E, R, H, M, A, ex, zp, sync, True, cmo)
    run_prequant(ep, cfg, idx, w, cmi)


def test_prequantised_prefill_full_size(ep):
    wl = W.WORKLOADS["prefill"]
    inp = W.make_inputs(wl, seed=0)
    cfg = HN.cfg_for(ep, wl)
    run_prequant(ep, cfg, inp["topk_idx"], inp["topk_weights"], col_major_input=True)


def test_prequantised_needs_an_fp8_handle(ep):
    idx, w = _routing(16, 2, 8, seed=1)
    cfg = ep.make_config(16, 2, 8, 2, 128, 8, 1, True, True, True, False)
    h = ep.ep_layout(cfg, idx.cuda())
    with pytest.raises(ep.EpError):
        ep.ep_dispatch_fp8(h, torch.zeros(16, 128, dtype=torch.uint8, device="cuda"),
                           torch.zeros(16, 1, device="cuda"), None,
                           torch.zeros(h.rows_alloc, 128, dtype=torch.uint8, device="cuda"),
                           torch.zeros(h.rows_alloc, device="cuda"))
    h.free()
