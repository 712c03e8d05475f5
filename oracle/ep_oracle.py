"""Plain, slow, obviously-correct CPU oracle for single-GPU MoE dispatch / combine.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg, never by the product path.  It shares no
code, table or helper with the CUDA library.

Sources (pages on DeepEP / vLLM; cited by title and section):

* "DeepEP V2 notes, ch. 7: how V2 dispatch builds expert inputs"
  - §7.1 input contract: ``topk_idx`` is [tokens, topk], -1 marks an empty
    slot; x is BF16 or an FP8 pair; ``topk_weights`` optional.
  - §7.2 layout metadata: the GPU produces receive counts, source metadata and
    slot indices; ``do_cpu_sync`` gives the exact size, otherwise the
    worst-case upper bound printed there (``num_max_tokens_per_rank *
    num_ranks`` received tokens; expanded rows ``num_ranks * M *
    min(topk, local_experts) + (alignment-1) * local_experts`` aligned).
  - §7.3 copy epilogue: rank layout or ``do_expand`` expert layout,
    ``expert_alignment`` pads each expert segment, ``do_zero_padding`` zeroes
    the gaps, FP8 scale factors may be stored TMA-aligned column-major.
  - §7.4 expanded layout: each expert owns one contiguous (padded) segment.
* "DeepEP V2 notes, ch. 8: combine, handle and async overlap", §8.1: combine
  reduces expert outputs back along the dispatch handle, with optional bias
  (``bias_0``, ``bias_1``) and top-k weights.
* "DeepEP README", interface example: ``get_dispatch_layout`` returns tokens
  per rank, tokens per expert and ``is_token_in_rank``.
* vLLM PR #52781 review, code excerpt of ``_finalize``: combine requires BF16
  input; the caller may pre-apply the weights and pass ``topk_weights=None``.

Where the pages leave a step open, the reading taken here is stated at the
function (R-numbers refer to the list of readings kept with the design notes).

Precision: the pages fix FP32 for the FP8 scale (scale = amax / 448) and for
the combine accumulation, so those steps are written in float32 numpy
arithmetic, one rounded operation per step (numpy never fuses a multiply and
an add).  Everything else is integer.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, library special cases, invariants).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "align", "upper_bound_rows", "layout", "bf16_bits_to_f32", "f32_to_bf16_bits",
    "e4m3_encode", "e4m3_decode", "quantize_row", "dispatch", "combine",
    "sf_numel", "sf_index", "FP8_BLOCK", "E4M3_MAX", "combine_topk_weights", "dispatch_prequantised",
    "layout_fixed_capacity",
]

FP8_BLOCK = 128        # 1x128 per-row scale blocks
E4M3_MAX = 448.0       # largest finite OCP E4M3FN value


def align(x, a):
    """Round up to a multiple of ``a`` (the pages' ``math::align``)."""
    return ((np.asarray(x, dtype=np.int64) + a - 1) // a) * a


# --------------------------------------------------------------------------
# Allocation sizes -- "V2 dispatch builds expert inputs" §7.2
# --------------------------------------------------------------------------
def upper_bound_rows(num_tokens, num_topk, num_experts, num_ranks, M, A, do_expand,
                     parts=False):
    """Rows the caller allocates when the host does not wait for the counts.

    §7.2 prints the per-rank worst case.  Reading R3: ranks are packed back to
    back in one allocation, so the total is ``min(R * per_rank, global)``,
    where the global bound is the most rows T tokens can ever produce.  The
    per-rank expression assumes a token names each expert at most once
    (``min(topk, local_experts)``); routing with repeated experts can exceed
    it, which ``layout`` reports as a capacity overflow.
    With ``parts=True`` returns ``(per_rank, global, rows)``.
    """
    T, K, E, R = num_tokens, num_topk, num_experts, num_ranks
    L = E // R
    if do_expand:
        per_rank = int(align(R * M * min(K, L) + (A - 1) * L, A))
        glob = int(align(T * K + E * (A - 1), A))
    else:
        per_rank = M * R
        glob = T * min(K, R)
    rows = min(R * per_rank, glob)
    return (per_rank, glob, rows) if parts else rows


def sf_numel(rows_alloc, hidden, col_major, capacity=None):
    """Number of fp32 scale slots the caller allocates for FP8 dispatch.

    ``capacity``: the fixed-capacity layout (``layout_fixed_capacity``), whose
    column-major scales are laid out per expert (reading R20)."""
    nb = hidden // FP8_BLOCK
    if col_major and capacity is not None:
        return (rows_alloc // capacity) * nb * int(align(capacity, 4))
    return nb * int(align(rows_alloc, 4)) if col_major else nb * rows_alloc


def sf_index(row, j, rows_alloc, hidden, col_major, capacity=None):
    """Flat index of scale block ``j`` of ``row``.

    Column-major TMA-aligned layout (§7.3): the hidden-block stride is the row
    count rounded up to 4 fp32 (16 bytes) -- reading R10.  In the
    fixed-capacity layout each expert's slab [capacity, H/128] is column-major
    on its own, with the row stride 1 and the block stride
    ``align(capacity, 4)`` (reading R20).  Row-major is ``row * H/128 + j``
    in every layout.
    """
    if col_major and capacity is not None:
        cap_al = int(align(capacity, 4))
        e, i = np.divmod(row, capacity)
        return e * (hidden // FP8_BLOCK) * cap_al + j * cap_al + i
    if col_major:
        return row + j * int(align(rows_alloc, 4))
    return row * (hidden // FP8_BLOCK) + j


# --------------------------------------------------------------------------
# Routing layout -- README get_dispatch_layout; §7.2; §7.4
# --------------------------------------------------------------------------
def layout(topk_idx, num_experts, num_ranks, num_max_tokens_per_rank,
           expert_alignment=1, do_expand=False, do_cpu_sync=True):
    """Counts, prefix sums, destination rows and source metadata.

    Definitions (experts are owned by ranks in contiguous blocks of
    L = E / R; token t comes from source rank t // M):

    * a slot (t, k) is valid iff topk_idx[t, k] != -1; any other value outside
      [0, E) is an error and the slot is treated as empty;
    * cnt_expert[e]     = number of valid slots routed to e;
    * cnt_expert_aligned= cnt_expert rounded up to the alignment A (R5);
    * psum_expert       = exclusive prefix of the aligned counts (E+1 entries);
    * is_token_in_rank  = token t has at least one valid slot on rank r;
    * cnt_rank[r]       = number of tokens with is_token_in_rank[t, r];
    * psum_rank         = exclusive prefix of cnt_rank (R+1 entries);
    * psum_rank_src[r]  = prefix over source ranks s of the tokens of s that
                          rank r receives (R x (R+1));
    * expanded layout: expert e's rows start at psum_expert[e]; inside the
      segment the slots are in ascending (t, k) order (reading R2); the
      remaining aligned rows are padding;
    * rank layout: one row per (token, rank) pair, rank r's rows start at
      psum_rank[r] and are in ascending token order; every slot of the token
      on that rank points to that row (R6), and the row's metadata names the
      lowest such slot.
    * capacity: without ``do_cpu_sync`` the rows live in an upper-bound
      allocation; a row at or past it (possible only with repeated experts in
      a token) is dropped -- its slots get destination -1 -- and the
      ``overflow`` error is raised.  Counts and prefix sums stay exact.

    ``error`` is a bit set: 1 = a topk_idx value outside [-1, E), 2 = overflow.
    """
    idx = np.array(topk_idx, dtype=np.int64, copy=True)
    if idx.ndim != 2:
        raise ValueError("topk_idx must be [tokens, topk]")
    T, K = idx.shape
    E, R, M, A = num_experts, num_ranks, num_max_tokens_per_rank, expert_alignment
    if E % R != 0 or A < 1 or M < 1 or T > M * R:
        raise ValueError("bad layout parameters")
    L = E // R

    bad = (idx < -1) | (idx >= E)
    error = 1 if bad.any() else 0
    idx[bad] = -1
    valid = idx >= 0
    rank_of = np.where(valid, idx // L, -1)

    cnt_expert = np.array([np.count_nonzero(idx == e) for e in range(E)], dtype=np.int64)
    cnt_expert_aligned = align(cnt_expert, A)
    psum_expert = np.concatenate([[0], np.cumsum(cnt_expert_aligned)]).astype(np.int64)

    in_rank = np.zeros((T, R), dtype=bool)
    for r in range(R):
        in_rank[:, r] = (rank_of == r).any(axis=1)
    cnt_rank = in_rank.sum(axis=0).astype(np.int64)
    psum_rank = np.concatenate([[0], np.cumsum(cnt_rank)]).astype(np.int64)

    src_rank = np.arange(T) // M
    psum_rank_src = np.zeros((R, R + 1), dtype=np.int64)
    for r in range(R):
        for s in range(R):
            got = int(np.count_nonzero(in_rank[src_rank == s, r]))
            psum_rank_src[r, s + 1] = psum_rank_src[r, s] + got

    num_expanded_tokens = int(psum_expert[E])
    num_recv_tokens = int(psum_rank[R])
    total_rows = num_expanded_tokens if do_expand else num_recv_tokens
    if do_cpu_sync:
        rows_alloc = total_rows
    else:
        rows_alloc = upper_bound_rows(T, K, E, R, M, A, do_expand)

    dst = np.full((T, K), -1, dtype=np.int64)
    meta = np.full((max(rows_alloc, total_rows), 2), -1, dtype=np.int64)
    flat_idx = idx.reshape(-1)
    flat_dst = dst.reshape(-1)
    if do_expand:
        for e in range(E):
            slots = np.flatnonzero(flat_idx == e)          # ascending (t, k)
            rows = psum_expert[e] + np.arange(slots.size)
            flat_dst[slots] = rows
            meta[rows, 0] = slots // K
            meta[rows, 1] = slots % K
    else:
        for r in range(R):
            toks = np.flatnonzero(in_rank[:, r])           # ascending t
            rows = psum_rank[r] + np.arange(toks.size)
            on_r = rank_of[toks] == r                      # [n, K]
            first_k = np.argmax(on_r, axis=1)              # lowest slot on r
            for k in range(K):
                sel = on_r[:, k]
                dst[toks[sel], k] = rows[sel]
            meta[rows, 0] = toks
            meta[rows, 1] = first_k

    if total_rows > rows_alloc:
        error |= 2
        dst[dst >= rows_alloc] = -1
    meta = meta[:rows_alloc]

    return {
        "T": T, "K": K, "E": E, "R": R, "L": L, "M": M, "A": A,
        "do_expand": bool(do_expand), "do_cpu_sync": bool(do_cpu_sync),
        "error": error,
        "topk_idx": idx,
        "cnt_expert": cnt_expert,
        "cnt_expert_aligned": cnt_expert_aligned,
        "psum_expert": psum_expert,
        "is_token_in_rank": in_rank,
        "cnt_rank": cnt_rank,
        "psum_rank": psum_rank,
        "psum_rank_src": psum_rank_src,
        "dst_buffer_slot_idx": dst,
        "recv_src_metadata": meta,
        "num_recv_tokens": num_recv_tokens,
        "num_expanded_tokens": num_expanded_tokens,
        "total_rows": total_rows,
        "rows_alloc": rows_alloc,
    }


def layout_fixed_capacity(topk_idx, num_experts, num_ranks, num_max_tokens_per_rank):
    """Fixed-capacity per-expert layout of the low-latency kernels (DeepEP
    README, "Interfaces and examples", low_latency_dispatch: per rank a
    [num_local_experts, num_max_dispatch_tokens_per_rank * num_ranks, hidden]
    receive tensor plus a per-expert count; CUDA-graph compatible).

    Reading R20: one GPU holds all R ranks' tensors back to back, so the rows
    form E slabs of ``capacity = M * R`` rows; expert e's i-th slot (slots in
    ascending (t, k), reading R2) lands at row ``e * capacity + i``.  Rows
    past a slab's count are unused (not written: unspecified).  No alignment
    padding.  A slot whose position reaches the capacity (possible only when
    a token repeats an expert) is dropped and raises the overflow error bit.
    Counts, rank outputs and prefix sums are those of ``layout`` with A = 1;
    ``rows_alloc = E * capacity`` whatever the counts are.
    """
    E, R, M = num_experts, num_ranks, num_max_tokens_per_rank
    lay = layout(topk_idx, E, R, M, 1, True, True)
    T, K = lay["T"], lay["K"]
    cap = M * R
    idx = lay["topk_idx"]
    rows_alloc = E * cap
    dst = np.full((T, K), -1, dtype=np.int64)
    meta = np.full((rows_alloc, 2), -1, dtype=np.int64)
    defined = np.zeros(rows_alloc, dtype=bool)
    error = lay["error"]
    flat_idx = idx.reshape(-1)
    flat_dst = dst.reshape(-1)
    for e in range(E):
        slots = np.flatnonzero(flat_idx == e)              # ascending (t, k)
        n = min(slots.size, cap)
        if slots.size > cap:
            error |= 2
        rows = e * cap + np.arange(n)
        flat_dst[slots[:n]] = rows
        meta[rows, 0] = slots[:n] // K
        meta[rows, 1] = slots[:n] % K
        defined[rows] = True
    lay = dict(lay)
    lay.update({
        "error": error, "dst_buffer_slot_idx": dst, "recv_src_metadata": meta,
        "rows_alloc": rows_alloc, "capacity": cap, "fixed_capacity": True,
        "row_defined": defined, "do_cpu_sync": False,
    })
    return lay


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------
def bf16_bits_to_f32(bits):
    """BF16 bit patterns (uint16) -> float32: the top half of an fp32 word."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(f):
    """float32 -> BF16 bits, round to nearest, ties to even; NaN stays NaN."""
    f = np.asarray(f, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
        r = np.where(nan, sign | np.uint16(0x7FC0), r)
    return r.astype(np.uint16)


def e4m3_encode(v):
    """float32 -> OCP FP8 E4M3FN byte, round to nearest even, saturating.

    Format (reading R8): 1 sign, 4 exponent (bias 7), 3 mantissa bits; normal
    values (1 + m/8) * 2^(e-7) for e in 1..15 (m <= 6 when e = 15), subnormals
    m * 2^-9; the largest finite value is 448; 0x7F / 0xFF are NaN; there is
    no infinity.  "satfinite": anything whose rounded magnitude exceeds 448,
    infinities included, becomes +-448; NaN becomes 0x7F (sign kept).
    """
    v = np.asarray(v, dtype=np.float32)
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.uint8)
    a = np.abs(v.astype(np.float64))
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.where(np.isinf(a), E4M3_MAX, a))
    _, ex = np.frexp(a)                      # a = m * 2^ex with m in [0.5, 1)
    e_unb = np.maximum(ex - 1, -6)           # floor(log2 a); subnormals use -6
    quantum = np.ldexp(1.0, e_unb - 3)       # 3 mantissa bits
    mag = np.rint(a / quantum) * quantum     # exact scaling, then RNE
    mag = np.minimum(mag, E4M3_MAX)
    m2, ex2 = np.frexp(mag)
    efield = ex2 - 1 + 7
    normal = (mag > 0) & (efield >= 1)
    mant_n = np.rint((m2 * 2.0 - 1.0) * 8.0)
    mant_s = np.rint(mag / 2.0 ** -9)
    code = np.where(normal, efield * 8 + mant_n, mant_s).astype(np.int64)
    code = np.where(nan, 0x7F, code).astype(np.uint8)
    return code | sign


def e4m3_decode(code):
    """OCP E4M3FN byte -> float64 (NaN for 0x7F/0xFF)."""
    c = np.asarray(code).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def quantize_row(x_bits):
    """One BF16 row -> (e4m3 bytes [H], fp32 scales [H/128]).

    Per 1x128 block j (reading R7): amax = max |x|; scale = amax / 448 in fp32
    (IEEE division, RNE); q = e4m3(x / scale) with an fp32 IEEE division
    (reading R8: a true division, not a multiply by 448 / amax).  An all-zero
    block has scale 0 and all bytes 0x00 (reading R9).

    Non-finite inputs (reading R16; the pages do not mention them): the amax
    propagates NaN, so a block holding a NaN has a NaN scale and every
    quotient is NaN; a block whose amax is infinite has scale +inf, its
    finite elements divide to +-0 and its infinite ones to NaN.  Every NaN
    quotient encodes as 0x7F, whatever the sign bit IEEE division left on
    it (that sign differs between hosts).
    """
    x = bf16_bits_to_f32(x_bits)
    H = x.shape[-1]
    if H % FP8_BLOCK:
        raise ValueError("hidden must be a multiple of 128 for FP8")
    blocks = x.reshape(*x.shape[:-1], H // FP8_BLOCK, FP8_BLOCK)
    amax = np.max(np.abs(blocks), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    zero = scale == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (blocks / np.where(zero, np.float32(1), scale)[..., None]).astype(np.float32)
    positive_nan = np.array([0x7FC00000], dtype=np.uint32).view(np.float32)[0]
    ratio = np.where(np.isnan(ratio), positive_nan, ratio)
    q = e4m3_encode(ratio)
    q = np.where(zero[..., None], np.uint8(0), q).astype(np.uint8)
    return q.reshape(x.shape), scale


# --------------------------------------------------------------------------
# Dispatch copy epilogue -- "V2 dispatch builds expert inputs" §7.3/§7.4
# --------------------------------------------------------------------------
def dispatch(lay, x_bits, topk_weights=None, use_fp8=False, col_major_sf=False,
             do_zero_padding=False):
    """Build every output of the copy epilogue on the CPU.

    Returns a dict with ``recv_x`` (BF16 bits [rows, H] or e4m3 bytes
    [rows, H]), ``recv_sf`` (flat fp32, FP8 only), ``recv_topk_weights``,
    ``recv_topk_idx`` (rank layout only) and boolean masks saying which rows
    the method defines (``payload_defined``, ``meta_defined``): rows past the
    total, and padding payload without ``do_zero_padding``, are unspecified.

    * every destination row gets a copy of its source token's row (BF16 bytes
      unchanged, or the FP8 bytes and scales of ``quantize_row``);
    * expanded layout: ``recv_topk_weights[row] = w[t, k]``; padding rows 0;
    * rank layout: ``recv_topk_weights[row, k] = w[t, k]`` and
      ``recv_topk_idx[row, k] = idx - r*L`` for the token's slots on rank r,
      0 and -1 for its other slots.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    if use_fp8:
        q, s = quantize_row(x_bits)
        return _scatter_rows(lay, q, s, topk_weights, col_major_sf, do_zero_padding)
    return _scatter_rows(lay, x_bits, None, topk_weights, False, do_zero_padding)


def dispatch_prequantised(lay, x_fp8, x_sf, topk_weights=None, col_major_sf=False,
                          do_zero_padding=False):
    """Dispatch of an input that is already FP8: ``x = (e4m3 bytes [T, H],
    fp32 scales [T, H/128])`` ("DeepEP V2 notes, ch. 7" §7.1 input contract,
    §7.3 copy epilogue).  Nothing is quantised: each destination row gets its
    token's bytes unchanged and its token's scales, written in the scale
    layout the handle asks for (row-major, or TMA-aligned column-major).
    Same outputs and masks as ``dispatch`` with ``use_fp8``."""
    q = np.asarray(x_fp8, dtype=np.uint8)
    s = np.asarray(x_sf, dtype=np.float32)
    assert q.ndim == 2 and s.shape == (q.shape[0], q.shape[1] // FP8_BLOCK)
    return _scatter_rows(lay, q, s, topk_weights, col_major_sf, do_zero_padding)


def _scatter_rows(lay, payload, scales, topk_weights, col_major_sf, do_zero_padding):
    """Copy each token's payload row (and scales) to its distinct rows, with
    the per-row weights and local expert ids; see ``dispatch``."""
    T, K, E, R, L = lay["T"], lay["K"], lay["E"], lay["R"], lay["L"]
    H = payload.shape[1]
    use_fp8 = scales is not None
    rows_alloc = lay["rows_alloc"]
    total = min(lay["total_rows"], rows_alloc)
    idx = lay["topk_idx"]
    dst = lay["dst_buffer_slot_idx"]
    rows = rows_alloc

    capacity = lay.get("capacity")
    payload_defined = np.zeros(rows, dtype=bool)
    if capacity is not None:
        payload_defined |= lay["row_defined"]
    else:
        payload_defined[:total] = True
    meta_defined = payload_defined.copy()
    padding = np.zeros(rows, dtype=bool)
    if lay["do_expand"] and capacity is None:
        pe, ce = lay["psum_expert"], lay["cnt_expert"]
        for e in range(E):
            padding[min(pe[e] + ce[e], rows):min(pe[e + 1], rows)] = True
        if not do_zero_padding:
            payload_defined &= ~padding

    if use_fp8:
        recv_x = np.zeros((rows, H), dtype=np.uint8)
        recv_sf = np.zeros(sf_numel(rows, H, col_major_sf, capacity), dtype=np.float32)
    else:
        recv_x = np.zeros((rows, H), dtype=np.uint16)
        recv_sf = None

    if lay["do_expand"]:
        recv_w = np.zeros(rows, dtype=np.float32)
        recv_i = None
    else:
        recv_w = np.zeros((rows, K), dtype=np.float32)
        recv_i = np.full((rows, K), -1, dtype=np.int32)

    nb = H // FP8_BLOCK
    for t in range(T):
        done = set()
        for k in range(K):
            row = int(dst[t, k])
            if row < 0 or row in done:
                continue
            done.add(row)
            recv_x[row] = payload[t]
            if use_fp8:
                for j in range(nb):
                    recv_sf[sf_index(row, j, rows, H, col_major_sf, capacity)] = scales[t, j]
            if lay["do_expand"]:
                if topk_weights is not None:
                    recv_w[row] = topk_weights[t, k]
            else:
                r = int(idx[t, k]) // L
                for kk in range(K):
                    if idx[t, kk] >= 0 and int(idx[t, kk]) // L == r:
                        if topk_weights is not None:
                            recv_w[row, kk] = topk_weights[t, kk]
                        recv_i[row, kk] = int(idx[t, kk]) - r * L
    return {
        "recv_x": recv_x, "recv_sf": recv_sf,
        "recv_topk_weights": recv_w, "recv_topk_idx": recv_i,
        "payload_defined": payload_defined, "meta_defined": meta_defined,
        "padding": padding,
    }


# --------------------------------------------------------------------------
# Combine -- "combine, handle and async overlap" §8.1; vLLM PR #52781
# --------------------------------------------------------------------------
def combine(lay, y_bits, topk_weights=None, bias_0=None, bias_1=None,
            expert_bias=None, tokens=None):
    """Weighted gather-reduce back to source-token order, fp32 -> BF16.

    For each token, ``acc = 0.0f``; for k = 0..K-1 in order, over valid slots:
    ``v = float(y[dst[t,k]])``; with a per-expert bias ``v = v + eb[idx]``
    (reading R13); ``acc = acc + w[t,k] * v`` (the product rounded to fp32,
    then the sum).  Without weights (reading R12) every slot counts with
    weight 1, but a row already used by an earlier slot of the same token is
    skipped.  Then ``acc += bias_0[t]``, ``acc += bias_1[t]``, and the result
    is rounded to BF16 (nearest even).  ``tokens`` restricts the computation to
    a subset of tokens (rows of the result follow that order).
    """
    idx = lay["topk_idx"]
    dst = lay["dst_buffer_slot_idx"]
    if tokens is None:
        tokens = np.arange(idx.shape[0])
    tokens = np.asarray(tokens, dtype=np.int64)
    idx, dst = idx[tokens], dst[tokens]
    K = idx.shape[1]
    y_bits = np.asarray(y_bits, dtype=np.uint16)
    H = y_bits.shape[1]
    n = tokens.size
    acc = np.zeros((n, H), dtype=np.float32)
    eb = None if expert_bias is None else bf16_bits_to_f32(expert_bias)
    w_all = None if topk_weights is None else np.asarray(topk_weights, np.float32)[tokens]
    for k in range(K):
        use = dst[:, k] >= 0
        if w_all is None:
            for kp in range(k):
                use &= ~((dst[:, kp] == dst[:, k]) & (dst[:, kp] >= 0))
            w = np.ones(n, dtype=np.float32)
        else:
            w = w_all[:, k]
        sel = np.flatnonzero(use)
        if sel.size == 0:
            continue
        v = bf16_bits_to_f32(y_bits[dst[sel, k]])
        if eb is not None:
            v = (v + eb[idx[sel, k]]).astype(np.float32)
        prod = (w[sel, None] * v).astype(np.float32)
        acc[sel] = (acc[sel] + prod).astype(np.float32)
    if bias_0 is not None:
        acc = (acc + bf16_bits_to_f32(np.asarray(bias_0)[tokens])).astype(np.float32)
    if bias_1 is not None:
        acc = (acc + bf16_bits_to_f32(np.asarray(bias_1)[tokens])).astype(np.float32)
    return f32_to_bf16_bits(acc)


# --------------------------------------------------------------------------
# Backward pair -- DeepEP README, "Interfaces and examples" (dispatch_backward
# is a combine of the received gradients together with their top-k weights;
# combine_backward is a dispatch of the combined gradient)
# --------------------------------------------------------------------------
def combine_topk_weights(lay, recv_topk_weights):
    """Reduction that combine applies to per-row top-k weights.

    The backward of dispatch is a combine that also carries the gradient of
    the received weights back to token order (DeepEP README, "Interfaces and
    examples", ``dispatch_backward``).  Reading R17: combine reduces the
    weights the way it reduces unweighted data -- a plain fp32 sum over the
    token's distinct destination rows, in the order the rows first appear in
    its slots.  Expanded layout: one scalar per row, and each row belongs to
    one slot, so slot k gets its own row's value (0 when the slot has no
    row).  Rank layout: ``recv_topk_weights`` is [rows, K]; the token's
    result is the sum of its rows' K-vectors, every column (0 for a token
    without rows).
    """
    dst = lay["dst_buffer_slot_idx"]
    T, K = dst.shape
    g = np.asarray(recv_topk_weights, dtype=np.float32)
    out = np.zeros((T, K), dtype=np.float32)
    for t in range(T):
        if lay["do_expand"]:
            for k in range(K):
                if dst[t, k] >= 0:
                    out[t, k] = g[dst[t, k]]
            continue
        seen = []
        for k in range(K):
            r = int(dst[t, k])
            if r >= 0 and r not in seen:
                seen.append(r)
        acc = np.zeros(K, dtype=np.float32)
        for r in seen:
            acc = (acc + g[r]).astype(np.float32)
        out[t] = acc
    return out
