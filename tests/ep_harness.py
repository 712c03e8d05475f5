"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
(Python binding) and compare every output with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import ep_workloads as W
from oracle import ep_oracle as O


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def cfg_for(ep, wl: W.Workload, T: int | None = None, **over):
    T = wl.num_tokens if T is None else T
    M = over.pop("M", max(wl.num_max_tokens_per_rank, -(-T // wl.num_ranks)))
    kw = dict(expert_alignment=wl.expert_alignment, do_expand=wl.do_expand,
              do_zero_padding=wl.do_zero_padding, do_cpu_sync=wl.do_cpu_sync,
              use_fp8=wl.use_fp8, use_tma_aligned_col_major_sf=wl.col_major_sf,
              fixed_capacity=wl.fixed_capacity)
    kw.update(over)
    return ep.make_config(T, wl.num_topk, wl.num_experts, wl.num_ranks, wl.hidden, M, **kw)


def oracle_layout(cfg, topk_idx: np.ndarray) -> dict:
    if getattr(cfg, "fixed_capacity", 0):
        return O.layout_fixed_capacity(topk_idx, cfg.num_experts, cfg.num_ranks,
                                       cfg.num_max_tokens_per_rank)
    return O.layout(topk_idx, cfg.num_experts, cfg.num_ranks, cfg.num_max_tokens_per_rank,
                    cfg.expert_alignment, bool(cfg.do_expand), bool(cfg.do_cpu_sync))


def gpu_layout_arrays(h) -> dict:
    torch.cuda.synchronize()
    names = ["topk_idx", "cnt_expert", "cnt_expert_aligned", "psum_expert", "cnt_rank",
             "psum_rank", "psum_rank_src", "dst_buffer_slot_idx", "recv_src_metadata",
             "is_token_in_rank", "totals", "error_word"]
    return {n: h.tensor(n).cpu().numpy() for n in names}


def check_layout(h, lay: dict, g: dict | None = None) -> dict:
    """Bit-exact comparison of every layout output."""
    g = gpu_layout_arrays(h) if g is None else g
    assert np.array_equal(g["topk_idx"], lay["topk_idx"]), "topk_idx copy"
    assert np.array_equal(g["cnt_expert"], lay["cnt_expert"]), "cnt_expert"
    assert np.array_equal(g["cnt_expert_aligned"], lay["cnt_expert_aligned"]), "aligned"
    assert np.array_equal(g["psum_expert"], lay["psum_expert"]), "psum_expert"
    assert np.array_equal(g["cnt_rank"], lay["cnt_rank"]), "cnt_rank"
    assert np.array_equal(g["psum_rank"], lay["psum_rank"]), "psum_rank"
    assert np.array_equal(g["psum_rank_src"], lay["psum_rank_src"]), "psum_rank_src"
    assert np.array_equal(g["is_token_in_rank"].astype(bool), lay["is_token_in_rank"]), "in_rank"
    assert np.array_equal(g["dst_buffer_slot_idx"], lay["dst_buffer_slot_idx"]), "dst"
    if "row_defined" in lay:     # fixed capacity: only each expert's used rows
        d = lay["row_defined"]
        assert np.array_equal(g["recv_src_metadata"][d], lay["recv_src_metadata"][d]), "meta"
    else:
        n = min(lay["total_rows"], lay["rows_alloc"])
        assert np.array_equal(g["recv_src_metadata"][:n], lay["recv_src_metadata"][:n]), "meta"
    assert g["totals"].tolist() == [lay["num_recv_tokens"], lay["num_expanded_tokens"]]
    assert int(g["error_word"][0]) == lay["error"], "error word"
    assert h.rows_alloc == lay["rows_alloc"], "rows_alloc"
    if h.cfg.do_cpu_sync:
        assert h.info.num_recv_tokens == lay["num_recv_tokens"]
        assert h.info.num_expanded_tokens == lay["num_expanded_tokens"]
    return g


def check_dispatch(h, lay: dict, d_or: dict, out: dict, use_fp8: bool, col_major: bool,
                   tokens: np.ndarray | None = None):
    """Bit-exact comparison of dispatch outputs on the rows the method defines.

    With ``tokens`` only the rows of those source tokens (and all padding rows)
    are compared; ``d_or`` then holds the oracle's per-token rows computed for
    exactly those tokens (see ``oracle_dispatch_tokens``)."""
    torch.cuda.synchronize()
    rows_alloc = lay["rows_alloc"]
    H = out["recv_x"].shape[1]
    if tokens is None:
        pdef = d_or["payload_defined"][:rows_alloc]
        if use_fp8:
            gx = out["recv_x"].cpu().numpy()
        else:
            gx = bits16(out["recv_x"])
        assert np.array_equal(gx[pdef], d_or["recv_x"][pdef]), "recv_x payload"
        if use_fp8:
            nb = H // 128
            gs = out["recv_sf"].cpu().numpy()
            rows = np.flatnonzero(pdef)
            for j in range(nb):
                ix = O.sf_index(rows, j, rows_alloc, H, col_major, lay.get("capacity"))
                # a block holding a NaN has a NaN scale (any payload, reading R16)
                assert np.array_equal(gs[ix], d_or["recv_sf"][ix], equal_nan=True), \
                    f"recv_sf block {j}"
        mdef = d_or["meta_defined"][:rows_alloc]
        if out.get("recv_topk_weights") is not None:
            gw = out["recv_topk_weights"].cpu().numpy()
            assert np.array_equal(gw[mdef], d_or["recv_topk_weights"][mdef]), "recv_topk_weights"
        if out.get("recv_topk_idx") is not None:
            gi = out["recv_topk_idx"].cpu().numpy()
            assert np.array_equal(gi[mdef], d_or["recv_topk_idx"][mdef]), "recv_topk_idx"
        return
    # sampled tokens at full size
    dst = lay["dst_buffer_slot_idx"]
    for i, t in enumerate(tokens):
        rows = sorted({int(r) for r in dst[t] if r >= 0})
        if not rows:
            continue
        ri = torch.tensor(rows, device=out["recv_x"].device)
        if use_fp8:
            gx = out["recv_x"].index_select(0, ri).cpu().numpy()
            assert np.all(gx == d_or["q"][i][None, :]), f"token {t} payload"
            nb = H // 128
            ix = np.stack([O.sf_index(np.array(rows), j, rows_alloc, H, col_major,
                                      lay.get("capacity"))
                           for j in range(nb)], 1)
            gs = out["recv_sf"][torch.from_numpy(ix.reshape(-1)).to(ri.device)].cpu().numpy()
            assert np.array_equal(gs.reshape(len(rows), nb),
                                  np.broadcast_to(d_or["s"][i], (len(rows), nb)),
                                  equal_nan=True), f"token {t} sf"
        else:
            gx = bits16(out["recv_x"].index_select(0, ri))
            assert np.all(gx == d_or["x"][i][None, :]), f"token {t} payload"


def oracle_dispatch_tokens(x_bits: np.ndarray, tokens: np.ndarray, use_fp8: bool) -> dict:
    if use_fp8:
        q, s = O.quantize_row(x_bits[tokens])
        return {"q": q, "s": s}
    return {"x": x_bits[tokens]}


def check_padding_zero(lay: dict, out: dict, use_fp8: bool, col_major: bool):
    """Property at any size: every alignment-padding row is zero (payload, scales)."""
    pe, ce = lay["psum_expert"], lay["cnt_expert"]
    rows_alloc = lay["rows_alloc"]
    rx = out["recv_x"]
    H = rx.shape[1]
    for e in range(lay["E"]):
        r0, r1 = int(pe[e] + ce[e]), int(min(pe[e + 1], rows_alloc))
        if r0 >= r1:
            continue
        blk = rx[r0:r1]
        assert int((blk.view(torch.uint8) != 0).sum()) == 0, f"padding payload expert {e}"
        if use_fp8:
            sf = out["recv_sf"]
            if col_major:
                st = -(-rows_alloc // 4) * 4
                v = sf.view(H // 128, st)[:, r0:r1]
            else:
                v = sf.view(rows_alloc, H // 128)[r0:r1]
            assert int((v != 0).sum()) == 0, f"padding sf expert {e}"


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)
