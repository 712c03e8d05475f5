"""GPU: one handle reused across dispatch modes, and independent handles
running concurrently on two streams, against the oracle.

A handle carries counters that its dispatches share (dynamic token and
padding scheduling, the column-major scale gather's handshake); every
dispatch must leave them ready for the next one, whatever the mode.
"""
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


def _routing(T, K, E, seed, drop=0.05):
    g = torch.Generator().manual_seed(seed)
    idx = torch.rand(T, E, generator=g).topk(K, dim=1).indices
    idx = idx.masked_fill(torch.rand(T, K, generator=g) < drop, -1)
    w = torch.rand(T, K, generator=g).masked_fill(idx < 0, 0.0)
    return idx.to(torch.int64).contiguous(), w.contiguous()


def _x(T, H, seed):
    return torch.randn(T, H, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)


@pytest.mark.parametrize("fixed", [False, True])
def test_one_handle_serves_every_dispatch_mode(ep, fixed):
    T, K, E, R, H, M = 1500, 8, 64, 8, 1024, 200
    idx, w = _routing(T, K, E, seed=5)
    if fixed:
        cfg = ep.make_config(T, K, E, R, H, M, 1, True, False, False, True, True,
                             fixed_capacity=True)
    else:
        cfg = ep.make_config(T, K, E, R, H, M, 16, True, True, True, True, True)
    h = ep.ep_layout(cfg, idx.cuda())
    lay = HN.oracle_layout(cfg, idx.numpy())
    HN.check_layout(h, lay)
    cm = True
    wd = w.cuda()
    for step, mode in enumerate(["quant", "prequant", "bf16", "quant", "quant", "prequant"]):
        if mode == "quant":
            x = _x(T, H, 10 + step)
            out = ep.alloc_recv(h, with_weights=True)
            ep.ep_dispatch(h, x.cuda(), wd, **out)
            d_or = O.dispatch(lay, HN.bits16(x), w.numpy(), True, cm, bool(cfg.do_zero_padding))
            HN.check_dispatch(h, lay, d_or, out, True, cm)
        elif mode == "prequant":
            g = torch.Generator().manual_seed(20 + step)
            xq = torch.randint(0, 256, (T, H), generator=g, dtype=torch.uint8)
            xs = torch.rand(T, H // 128, generator=g)
            out = ep.alloc_recv(h, with_weights=True)
            ep.ep_dispatch_fp8(h, xq.cuda(), xs.cuda(), wd, **out)
            d_or = O.dispatch_prequantised(lay, xq.numpy(), xs.numpy(), w.numpy(), cm,
                                           bool(cfg.do_zero_padding))
            HN.check_dispatch(h, lay, d_or, out, True, cm)
        else:
            x = _x(T, H, 30 + step)
            got = ep.ep_combine_backward(h, x.cuda())
            torch.cuda.synchronize()
            d_or = O.dispatch(lay, HN.bits16(x), None, False, False, bool(cfg.do_zero_padding))
            pdef = d_or["payload_defined"][:h.rows_alloc]
            assert np.array_equal(HN.bits16(got)[pdef], d_or["recv_x"][pdef]), f"step {step}"
        # no dispatch of this handle may leave the device error word set
        assert int(h.tensor("error_word").cpu()[0]) == lay["error"], f"step {step} ({mode})"
    h.free()


def test_independent_handles_on_two_streams(ep):
    """Two full paths (layout, dispatch, combine) enqueued alternately on two
    streams, without host synchronisation, both checked against the oracle."""
    T, K, E, R, H, M = 2000, 8, 64, 8, 1024, 250
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    cases = []
    for j in range(2):
        idx, w = _routing(T, K, E, seed=40 + j)
        cfg = ep.make_config(T, K, E, R, H, M, 8, True, True, False, True, True)
        x = _x(T, H, 50 + j)
        cases.append((cfg, idx, w, x))
    dev = [(idx.cuda(), w.cuda(), x.cuda()) for _, idx, w, x in cases]
    torch.cuda.synchronize()
    handles, outs, ys, res = [], [], [], []
    for j, (cfg, idx, w, x) in enumerate(cases):
        with torch.cuda.stream(streams[j]):
            h = ep.ep_layout(cfg, dev[j][0], stream=streams[j])
            handles.append(h)
    for j, (cfg, idx, w, x) in enumerate(cases):
        with torch.cuda.stream(streams[j]):
            out = ep.alloc_recv(handles[j], with_weights=True)
            ep.ep_dispatch(handles[j], dev[j][2], dev[j][1], stream=streams[j], **out)
            outs.append(out)
    for j, (cfg, idx, w, x) in enumerate(cases):
        with torch.cuda.stream(streams[j]):
            rows = handles[j].rows_alloc
            y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
            for r0 in range(0, rows, 8192):
                r1 = min(rows, r0 + 8192)
                y[r0:r1] = W.hashed_bf16_rows(torch.arange(r0, r1, device="cuda"), H, 60 + j, "cuda")
            ys.append(y)
            res.append(ep.ep_combine(handles[j], y, dev[j][1], stream=streams[j]))
    torch.cuda.synchronize()
    for j, (cfg, idx, w, x) in enumerate(cases):
        lay = HN.oracle_layout(cfg, idx.numpy())
        HN.check_layout(handles[j], lay)
        d_or = O.dispatch(lay, HN.bits16(x), w.numpy(), True, True, True)
        HN.check_dispatch(handles[j], lay, d_or, outs[j], True, True)
        rows = handles[j].rows_alloc
        need = np.unique(lay["dst_buffer_slot_idx"])
        need = need[need >= 0]
        y_bits = np.zeros((rows, H), dtype=np.uint16)
        y_bits[need] = HN.bits16(W.hashed_bf16_rows(torch.from_numpy(need), H, 60 + j))
        ref = O.combine(lay, y_bits, w.numpy())
        d = HN.ulp_diff(HN.bits16(res[j]), ref)
        assert d.max(initial=0) <= 1
        handles[j].free()


@pytest.mark.parametrize("expand", [False, True])
def test_repeated_combines_on_one_handle(ep, expand):
    """Back-to-back combines and dispatch_backward calls on one handle, with
    the expert bias on and off: each gives what the oracle gives (nothing a
    combine leaves behind changes the next one)."""
    T, K, E, R, H, M = 3000, 6, 32, 4, 512, 750
    idx, w = _routing(T, K, E, seed=41)
    cfg = ep.make_config(T, K, E, R, H, M, 8 if expand else 1, expand, expand, True)
    h = ep.ep_layout(cfg, idx.cuda())
    lay = HN.oracle_layout(cfg, idx.numpy())
    rows = h.rows_alloc
    eb = W.hashed_bf16_rows(torch.arange(E), H, 77)
    w_np = w.numpy()
    for rep in range(3):
        y = W.hashed_bf16_rows(torch.arange(rows), H, 50 + rep)
        y_bits = HN.bits16(y)
        use_eb = rep % 2 == 1
        got = ep.ep_combine(h, y.cuda(), w.cuda(), None, None, eb.cuda() if use_eb else None)
        ref = O.combine(lay, y_bits, w_np, None, None, HN.bits16(eb) if use_eb else None)
        assert HN.ulp_diff(HN.bits16(got), ref).max(initial=0) == 0, rep
        gx = ep.ep_dispatch_backward(h, y.cuda(), None)[0]
        ref_b = O.combine(lay, y_bits, None, None, None, None)
        assert HN.ulp_diff(HN.bits16(gx), ref_b).max(initial=0) == 0, rep
    h.free()
