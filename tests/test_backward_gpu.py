"""GPU parity of the backward pair (DeepEP README, "Interfaces and examples":
dispatch_backward is a combine that also reduces the weight gradients,
combine_backward is a dispatch of the gradient) against the CPU oracle.

combine_backward copies BF16 bytes: bit-exact.  The weight reduction rounds
every add like the oracle: bit-exact.  The data part of dispatch_backward is
the unweighted combine: within 1 BF16 ulp (in practice bit-exact).
"""
import zlib

import numpy as np
import pytest
import torch

import ep_workloads as W
from oracle import ep_oracle as O
from tests import ep_harness as HN

pytestmark = pytest.mark.gpu

COMBINE_ULP = 1


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
    return idx.to(torch.int64).contiguous()


def check_backward(ep, cfg, idx_cpu, *, seed=21, tokens=None):
    """Runs both backward entry points on one handle and compares with the
    oracle; ``tokens`` restricts the data comparison of dispatch_backward to
    a sample of tokens (full-size cases)."""
    dev = torch.device("cuda")
    T, K, H = cfg.num_tokens, cfg.num_topk, cfg.hidden
    h = ep.ep_layout(cfg, idx_cpu.to(dev))
    lay = HN.oracle_layout(cfg, idx_cpu.to(torch.int64).numpy())
    HN.check_layout(h, lay)
    rows = h.rows_alloc

    # combine_backward: BF16 dispatch of the gradient, whatever cfg.use_fp8 says
    g_out = W.hashed_bf16_rows(torch.arange(T, device=dev), H, seed, dev)
    canary = 3
    buf = torch.full((rows + canary, H), -1.5, dtype=torch.bfloat16, device=dev)
    ep.ep_combine_backward(h, g_out, buf[:rows] if rows else buf[:0])
    torch.cuda.synchronize()
    d_or = O.dispatch(lay, HN.bits16(g_out), None, False, False, bool(cfg.do_zero_padding))
    pdef = d_or["payload_defined"][:rows]
    gx = HN.bits16(buf[:rows])
    assert np.array_equal(gx[pdef], d_or["recv_x"][pdef]), "combine_backward rows"
    assert bool((buf[rows:] == -1.5).all()), "combine_backward wrote past rows_alloc"

    # dispatch_backward: unweighted combine of grad_recv_x + the weight reduction
    grad_recv = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, rows, 8192):
        r1 = min(rows, r0 + 8192)
        grad_recv[r0:r1] = W.hashed_bf16_rows(torch.arange(r0, r1, device=dev), H, seed + 1, dev)
    gshape = (rows,) if cfg.do_expand else (rows, K)
    gw = torch.randn(gshape, generator=torch.Generator().manual_seed(seed + 2)).to(dev)
    gw_out = torch.full((T * K + canary,), 7.25, device=dev)
    gx_out, gw_ret = ep.ep_dispatch_backward(h, grad_recv, gw, grad_topk_weights=gw_out[:T * K]
                                             .view(T, K))
    torch.cuda.synchronize()
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    need = np.unique(lay["dst_buffer_slot_idx"][toks])
    need = need[need >= 0]
    y_bits = np.zeros((max(rows, 1), H), dtype=np.uint16)
    if need.size:
        y_bits[need] = HN.bits16(W.hashed_bf16_rows(torch.from_numpy(need), H, seed + 1))
    ref = O.combine(lay, y_bits, None, tokens=toks)
    got = HN.bits16(gx_out.index_select(0, torch.from_numpy(toks).to(dev)))
    d = HN.ulp_diff(got, ref)
    assert d.max(initial=0) <= COMBINE_ULP, f"dispatch_backward max ulp {d.max(initial=0)}"
    ref_w = O.combine_topk_weights(lay, gw.cpu().numpy())
    got_w = gw_ret.cpu().numpy()
    assert np.array_equal(got_w.view(np.uint32), ref_w.view(np.uint32)), "grad_topk_weights"
    assert bool((gw_out[T * K:] == 7.25).all()), "weight reduction wrote past [T, K]"
    # without weight gradients only grad_x is produced
    gx2, none = ep.ep_dispatch_backward(h, grad_recv)
    assert none is None
    torch.cuda.synchronize()
    assert torch.equal(gx2, gx_out)
    h.free()
    return int((d != 0).sum())


CASES = {
    # name: (T, K, E, R, H, M, A, expand, zero_pad, sync, fp8, col_major, drop, dup)
    "expand_fp8_cfg": (700, 8, 64, 8, 256, 100, 16, True, True, True, True, True, 0.1, False),
    "expand_no_zero_pad": (300, 4, 16, 4, 128, 75, 8, True, False, True, False, False, 0.1, False),
    "rank_layout": (513, 8, 64, 8, 512, 65, 1, False, False, True, False, False, 0.1, False),
    "rank_dup_experts": (200, 6, 8, 2, 128, 100, 1, False, False, True, False, False, 0.1, True),
    "expand_dup_experts": (200, 6, 8, 2, 128, 100, 4, True, True, True, False, False, 0.1, True),
    "rank_nosync": (600, 8, 32, 8, 256, 75, 1, False, False, False, True, False, 0.0, False),
    "expand_nosync": (600, 8, 32, 8, 256, 75, 8, True, True, False, False, False, 0.0, False),
    "all_slots_empty": (40, 3, 8, 4, 64, 10, 4, True, True, True, False, False, 1.0, False),
    "empty_tokens": (0, 4, 8, 2, 64, 4, 4, True, True, True, False, False, 0.0, False),
    "max_topk": (64, 32, 64, 4, 128, 16, 4, False, False, True, False, False, 0.0, False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_pair(ep, case):
    T, K, E, R, H, M, A, ex, zp, sync, fp8, cm, drop, dup = CASES[case]
    idx = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop, dup=dup)
    cfg = ep.make_config(T, K, E, R, H, M, A, ex, zp, sync, fp8, cm)
    assert check_backward(ep, cfg, idx) == 0


def test_backward_overflow_dropped_rows(ep):
    """Rows past the allocation are dropped on both passes (their slots read
    no row and get weight gradient 0)."""
    idx = torch.tensor([[0, 0, 0, 0], [1, 1, 0, 0]], dtype=torch.int64)
    cfg = ep.make_config(2, 4, 2, 2, 128, 1, 1, True, True, False, False, False)
    assert check_backward(ep, cfg, idx) == 0


@pytest.mark.parametrize("name", ["prefill", "decode", "skewed"])
def test_backward_full_size(ep, name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl, seed=0)
    cfg = HN.cfg_for(ep, wl)
    T = wl.num_tokens
    rng = np.random.default_rng(4)
    toks = np.sort(rng.choice(T, size=min(T, 256), replace=False))
    assert check_backward(ep, cfg, inp["topk_idx"], tokens=toks) == 0
