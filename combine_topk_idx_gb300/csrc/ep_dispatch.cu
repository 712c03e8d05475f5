// Dispatch copy epilogue: source rows -> rank layout or expert-expanded layout.
//
// Follows "DeepEP V2 notes, ch. 7: how V2 dispatch builds expert inputs",
// §7.3 (copy epilogue: expand / rank layout, expert_alignment padding,
// do_zero_padding, TMA-aligned column-major scale factors) and §7.4; the FP8
// payload is e4m3 with one fp32 scale per 1x128 block (scale = amax / 448).
//
// Token-major scatter with persistent, warp-specialised CTAs:
//   warp 0 (producer) takes tokens -- CTA b's first S are b, b + G, ...
//     (G CTAs, S stages), then the next free one from a handle counter --
//     issues one cp.async.bulk global->shared copy of the token's source row
//     into a ring of input stages (S = 3; 2 for quantised rows too large for
//     three; the stage's "full" barrier counts the bytes), then reads the
//     token's K destination rows (fetched while the previous token was
//     issued), keeps the distinct ones (rank-layout slots of one rank share a
//     row), writes the per-row weights and local expert ids and arrives on
//     the stage's "rows" barrier;
//   the consumer warps wait for a stage's "full" barrier and
//     FP8:  quantise it -- amax of each 128-element block by a 16-lane
//           shuffle, scale = amax / 448 (IEEE division) and the e4m3 bytes of
//           x / scale (packed cvt.rn.satfinite.e4m3x2 of a bracket of the
//           quotient, IEEE quotients wherever the bracket straddles a
//           rounding boundary) -- into an output stage, then, once "rows"
//           completes, one thread issues one cp.async.bulk shared->global
//           store per distinct destination row while the others write the
//           scales;
//     BF16: one thread stores the input stage itself to every row;
//     pre-quantised FP8 input (x given as e4m3 bytes + fp32 scales, §7.1):
//           the same copy of the H-byte row, while the other threads copy
//           the token's scales to each row (row-major) or leave them to the
//           column-major gather, which then reads the caller's scales.
// The source row is read from HBM once and quantised once whatever K is; the
// TMA engine moves every payload byte.  After the tokens, the consumer warps
// zero the alignment padding rows in 8-row work items, also handed out from a
// handle counter.  The kernel is launched with programmatic dependent
// launch: nothing reads the layout's outputs before griddepcontrol.wait; with
// early_x (the layout was launched by the same call, so x was complete before
// it) the first S source rows are loaded, and quantised, before the wait.
// Every mbarrier wait is bounded: a wait that gives up sets EP_ERRBIT_TIMEOUT
// and the CTA returns.
#include <algorithm>

#include "ep_internal.cuh"
#include "ep_ptx.cuh"

namespace ep {
namespace {

constexpr int kStages = 3;              // stage ring depth (2: see launch_one)
constexpr int kFewTokens = 8192;        // quantising up to this many tokens: two stages
constexpr size_t kSmemLimit = 227 * 1024 - 4096;  // dynamic share, static arrays set aside
constexpr int kPadRowsPerItem = 8;
constexpr int kMaxConsumers = 224;
constexpr int kWaitIters = 4000;          // x kWaitHintNs: gives up after ~2 s
constexpr uint32_t kWaitHintNs = 500000;
constexpr int kBarConsumers = 1;          // named barrier id (0 is __syncthreads)
constexpr int kSfRowsPerThread = 4;       // scale gather: rows per thread
constexpr int kSfWaitIters = 8000000;     // x ~256 ns: the gather gives up after ~2 s
// What the scale gather waits for before reading per-token scales.
constexpr int kSfWaitNone = 0;            // nothing: the caller's scales (pre-quantised)
constexpr int kSfWaitHandshake = 1;       // every dispatch CTA's published counter
constexpr int kSfWaitGrid = 2;            // the whole dispatch grid (griddepcontrol.wait)

// What the kernel does with a source row.
constexpr int kModeBf16 = 0;    // BF16 in, BF16 copy out
constexpr int kModeQuant = 1;   // BF16 in, quantised to e4m3 + fp32 scales
constexpr int kModePreq = 2;    // e4m3 + fp32 scales in, copied

struct TokenMeta {
  int rows[EP_MAX_TOPK];
  int n;
  int t;  // source token, or -1: no more tokens for this CTA
};

// Expert whose padding range holds padding row q: the last e with psum_pad[e] <= q.
__device__ __forceinline__ int padding_expert(const int32_t *psum_pad, int E, int q) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(psum_pad + mid) <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One work item of alignment padding: up to kPadRowsPerItem consecutive
// padding rows (numbered across all experts): zero payload, scales, weight.
// Run by the consumer threads only (ctid in [0, nct)).
__device__ __forceinline__ void zero_padding_item(const DispatchParams &p, int item, int npad,
                                                  int *prow, bool fp8, bool col_major, int ctid,
                                                  int nct) {
  const int q0 = item * kPadRowsPerItem;
  if (ctid < kPadRowsPerItem) {
    const int q = q0 + ctid;
    int64_t row = -1;
    if (q < npad) {
      const int e = padding_expert(p.psum_pad, p.E, q);
      row = (int64_t)__ldg(p.psum_e + e) + __ldg(p.cnt_e + e) + (q - __ldg(p.psum_pad + e));
      if (row >= p.rows_alloc) row = -1;
    }
    prow[ctid] = (int)row;
  }
  named_barrier(kBarConsumers, nct);
  if (p.recv_w != nullptr && ctid < kPadRowsPerItem && prow[ctid] >= 0) p.recv_w[prow[ctid]] = 0.f;
  if (!p.zero_padding) return;
  const int64_t row_bytes = fp8 ? p.H : 2 * (int64_t)p.H;
  const int n16 = (int)(row_bytes / 16);
  const uint4 z = make_uint4(0, 0, 0, 0);
  uint8_t *recv = static_cast<uint8_t *>(p.recv_x);
  for (int i = ctid; i < kPadRowsPerItem * n16; i += nct) {
    const int r = i / n16;
    const int row = prow[r];
    if (row >= 0) st_stream_v4(recv + (int64_t)row * row_bytes + (int64_t)(i - r * n16) * 16, z);
  }
  if (fp8 && !col_major) {  // column-major padding scales are zeroed by the scale gather
    const int nb = p.H / kFp8Block;
    for (int i = ctid; i < kPadRowsPerItem * nb; i += nct) {
      const int r = i / nb;
      const int row = prow[r];
      if (row >= 0) p.recv_sf[(int64_t)row * nb + (i - r * nb)] = 0.f;
    }
  }
}

struct Routing {
  int d, e;
  float w;
};

// e4m3 bytes of x / sc for eight elements (f: x as fp32), equal to the
// round-to-nearest-even, saturating conversion of the IEEE fp32 quotients.
// With r the reciprocal of sc within 2 ulp (relative error 2^-22), the
// products x * r * (1 -+ 2^-17), each rounded, bracket the rounded quotient
// strictly (every rounding error is below 2^-21 of the 2^-17 margin).  The
// conversion is monotonic in the magnitude, so where both ends of the
// bracket convert to the same byte, the quotient does too; where they differ
// -- a rounding boundary of the e4m3 grid inside the bracket, about 1 element
// in 200 of BF16 data, mostly exact ties -- that pair of quotients is taken
// by IEEE division (per pair, so a warp runs the divisions only for pairs
// where some lane needs them).  Outside sc in [2^-120, 2^120) the reciprocal
// loses its accuracy and every quotient is a division.
__device__ __forceinline__ uint2 e4m3_block8(const float *f, float sc) {
  const uint32_t sb = __float_as_uint(sc);
  uint32_t c[4];
  if (sb >= 0x03800000u && sb < 0x7B800000u) {
    const float r = __fdividef(1.0f, sc);
    const float rl = r * 0.99999237060546875f, rh = r * 1.00000762939453125f;  // 1 -+ 2^-17
    const uint64_t rl2 = f32x2_pack(rl, rl), rh2 = f32x2_pack(rh, rh);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t x2 = f32x2_pack(f[2 * q], f[2 * q + 1]);
      const uint64_t lo = f32x2_mul_rn(x2, rl2), hi = f32x2_mul_rn(x2, rh2);
      c[q] = cvt_e4m3x2(f32x2_lo(lo), f32x2_hi(lo));
      if (c[q] != cvt_e4m3x2(f32x2_lo(hi), f32x2_hi(hi)))
        c[q] = cvt_e4m3x2(__fdiv_rn(f[2 * q], sc), __fdiv_rn(f[2 * q + 1], sc));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      c[q] = cvt_e4m3x2(__fdiv_rn(f[2 * q], sc), __fdiv_rn(f[2 * q + 1], sc));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ Routing load_routing(const DispatchParams &p, int t, int lane) {
  Routing r{-1, -1, 0.f};
  if (lane < p.K) {
    const int64_t o = (int64_t)t * p.K + lane;
    r.d = __ldg(p.dst + o);
    r.e = __ldg(p.topk32 + o);
    if (p.topk_w != nullptr) r.w = __ldg(p.topk_w + o);
  }
  return r;
}

template <int MODE, bool COL_MAJOR, int S>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) dispatch_kernel(DispatchParams p) {
  constexpr bool FP8 = MODE == kModeQuant;         // quantise in the consumers
  constexpr bool FP8_OUT = MODE != kModeBf16;      // e4m3 payload + scales
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[S];    // source row landed (and meta[s].t set)
  __shared__ __align__(8) uint64_t rows[S];    // row list of the stage written
  __shared__ __align__(8) uint64_t empty[S];
  __shared__ TokenMeta meta[S];
  __shared__ int prow_s[2][kPadRowsPerItem];

  const int H = p.H;
  const int in_bytes = MODE == kModePreq ? H : 2 * H;     // source row
  const int in_stage = (in_bytes + 127) / 128 * 128;
  const int out_bytes = FP8_OUT ? H : 2 * H;               // destination row
  const int out_stage = FP8 ? (H + 127) / 128 * 128 : 0;
  const int nb = H / kFp8Block;
  const int nb_pad = (nb + 31) / 32 * 32;
  uint8_t *in0 = smem;
  uint8_t *out0 = smem + S * in_stage;
  float *sf0 = reinterpret_cast<float *>(out0 + S * out_stage);  // row-major scales
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncw = (blockDim.x >> 5) - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&rows[s], 1);
      mbar_init(&empty[s], ncw);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // x rows and the destination payload are touched once: evict them first so
  // that the small, scattered scale-factor sectors stay in L2 until complete.
  const uint64_t stream_pol = l2_policy_evict_first();
  auto issue_row = [&](int s, int t) {  // lane 0 of the producer
    meta[s].t = t;
    mbar_arrive_expect_tx(&full[s], (uint32_t)in_bytes);
    const void *src = MODE == kModePreq ? static_cast<const void *>(p.xq + (int64_t)t * H)
                                        : static_cast<const void *>(p.x + (int64_t)t * H);
    bulk_load_g2s_hint(in0 + s * in_stage, src, (uint32_t)in_bytes, &full[s], stream_pol);
  };
  if (warp == 0) {
    // ---------------- producer ----------------
    // CTA b's first S tokens are b, b + G, ..., b + (S - 1) G; the rest are
    // handed out dynamically from a handle counter, so CTAs that run faster
    // take more of them.  The next token and its routing are fetched while
    // the current one is issued.
    const int G = gridDim.x;
    // Launched with programmatic dependent launch: everything above overlaps
    // the tail of the kernel before this one.  The first S source rows need
    // no output of that kernel; with early_x their loads leave before the
    // wait.  Nothing below the wait reads global memory before that kernel's
    // writes are visible.
    const int64_t early = p.early_x ? S : 0;
    if (lane == 0)
      for (int k = 0; k < early && blockIdx.x + (int64_t)k * G < p.T; ++k)
        issue_row(k, (int)(blockIdx.x + (int64_t)k * G));
    griddep_wait();
    int next = blockIdx.x;
    Routing rn{-1, -1, 0.f};
    if (next < p.T) rn = load_routing(p, next, lane);
    for (int64_t i = 0;; ++i) {
      const int t = next;
      const int s = (int)(i % S);
      const int64_t k = i / S;
      if (k > 0) {
        bool ok = false;
        if (lane == 0)
          ok = mbar_wait_bounded(&empty[s], (uint32_t)((k - 1) & 1), kWaitIters, kWaitHintNs);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) atomicOr(p.err, EP_ERRBIT_TIMEOUT);
          return;
        }
      }
      if (t >= p.T) {  // end marker for the consumers
        if (lane == 0) {
          meta[s].t = -1;
          mbar_arrive(&full[s]);
        }
        break;
      }
      const Routing cur = rn;
      // The source row first (unless it left before the wait): its load
      // needs only the token index, so it overlaps the ticket for the next
      // token and the routing work below.
      if (lane == 0) {
        if (i >= early) issue_row(s, t);
        next = i + 1 < S ? (int)min((int64_t)p.T, blockIdx.x + (i + 1) * (int64_t)G)
                         : S * G + atomicAdd(p.sched, 1);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, cur.d);
      const bool keep = cur.d >= 0 && lane == __ffs(peers) - 1;
      const unsigned keepm = __ballot_sync(0xffffffffu, keep);
      const int n = __popc(keepm);
      if (keep) meta[s].rows[__popc(keepm & lanemask_lt())] = cur.d;
      if (lane == 0) {
        meta[s].n = n;
        meta[s].t = t;
      }
      if (p.do_expand) {
        if (keep && p.recv_w != nullptr) p.recv_w[cur.d] = cur.w;
      } else if (p.recv_w != nullptr || p.recv_idx != nullptr) {
        // lane kk < K holds slot kk: its rank and local expert id once; then
        // for each kept row, the K lanes write its K entries side by side
        const int my_r = cur.e >= 0 ? cur.e / p.L : -1;
        const int my_l = cur.e - my_r * p.L;
        for (unsigned m = keepm; m; m &= m - 1) {
          const int src = __ffs(m) - 1;
          const int row = __shfl_sync(0xffffffffu, cur.d, src);
          const int rr = __shfl_sync(0xffffffffu, my_r, src);
          if (lane < p.K) {
            const bool same = my_r >= 0 && my_r == rr;
            const int64_t o = (int64_t)row * p.K + lane;
            if (p.recv_w != nullptr) p.recv_w[o] = same ? cur.w : 0.f;
            if (p.recv_idx != nullptr) p.recv_idx[o] = same ? my_l : -1;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rows[s]);
      next = __shfl_sync(0xffffffffu, next, 0);
      if (next < p.T) rn = load_routing(p, next, lane);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = threadIdx.x - 32;
  const int nct = blockDim.x - 32;
  const int nvec = H / 8;  // 16-byte vectors of the BF16 row
  uint8_t *recv = static_cast<uint8_t *>(p.recv_x);
  // Quantising a row needs only the row itself; its row list (the layout's
  // output) is read after the wait.
  bool waited = false;
  // row-major scale stores: when nb divides the consumer count, thread ctid
  // owns scale column ctid % nb of rows ctid / nb, + nct / nb, ...
  const int sf_step = (nb > 0 && nct % nb == 0) ? nct / nb : 0;
  const int sf_j = sf_step > 0 ? ctid % nb : 0;
  const int sf_r0 = sf_step > 0 ? ctid / nb : 0;
  for (int64_t i = 0;; ++i) {
    const int s = (int)(i % S);
    const uint32_t par = (uint32_t)((i / S) & 1);
    auto wait_or_fail = [&](uint64_t *bar) {
      if (mbar_wait_bounded(bar, par, kWaitIters, kWaitHintNs)) return true;
      if (!waited) griddep_wait();
      if (lane == 0) atomicOr(p.err, EP_ERRBIT_TIMEOUT);
      if (ctid == 0) bulk_wait_all<0>();
      return false;
    };
    if (!wait_or_fail(&full[s])) return;
    const int t = meta[s].t;
    if (t < 0) break;  // the producer has no more tokens
    const uint8_t *in = in0 + s * in_stage;
    if constexpr (FP8) {
      uint8_t *out = out0 + s * out_stage;
      float *sf = sf0 + s * nb_pad;
      // out stage s no longer read: at most S - 1 later bulk groups pending
      if (ctid == 0) bulk_wait_read<S - 1>();
      named_barrier(kBarConsumers, nct);
      // every consumer thread runs the same number of iterations so the
      // 16-lane shuffles always see full warps (nvec and nct are multiples of 16)
      for (int v0 = 0; v0 < nvec; v0 += nct) {
        const int v = v0 + ctid;
        const bool valid = v < nvec;
        const uint4 x8 = valid ? *reinterpret_cast<const uint4 *>(in + v * 16)
                               : make_uint4(0, 0, 0, 0);
        float f[8];
        f[0] = bf16_lo(x8.x); f[1] = bf16_hi(x8.x);
        f[2] = bf16_lo(x8.y); f[3] = bf16_hi(x8.y);
        f[4] = bf16_lo(x8.z); f[5] = bf16_hi(x8.z);
        f[6] = bf16_lo(x8.w); f[7] = bf16_hi(x8.w);
        // amax propagates NaN (max.NaN): a block holding a NaN gets a NaN
        // scale and the NaN code 0x7F in every byte
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) amax = fmax_nan(amax, fabsf(f[q]));
        // 16 consecutive lanes hold one 128-element block
        amax = fmax_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmax_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmax_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        amax = fmax_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
        if (valid) {
          const float sc = __fdiv_rn(amax, 448.0f);
          uint2 packed = make_uint2(0, 0);
          if (amax != amax) {
            packed = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
          } else if (amax != 0.f) {
            // an infinite amax: finite elements divide to +-0, infinite ones
            // to NaN, which the conversion encodes as 0x7F
            packed = e4m3_block8(f, sc);
          }
          *reinterpret_cast<uint2 *>(out + v * 8) = packed;
          if ((v & 15) == 0) {
            if (COL_MAJOR)
              p.tok_scale[(int64_t)t * nb + (v >> 4)] = sc;
            else
              sf[v >> 4] = sc;
          }
        }
      }
      fence_proxy_async_smem();
      if (!waited) {
        griddep_wait();
        waited = true;
      }
      if (!wait_or_fail(&rows[s])) return;
      const int n = meta[s].n;
      named_barrier(kBarConsumers, nct);
      if (ctid == 0) {
        for (int r = 0; r < n; ++r)
          bulk_store_s2g_hint(recv + (int64_t)meta[s].rows[r] * out_bytes, out, (uint32_t)out_bytes,
                              stream_pol);
        bulk_commit();  // one bulk group per token (empty when n = 0) keeps the stage reuse exact
      }
      if (!COL_MAJOR) {  // row-major scales: nb contiguous floats per row
        if (sf_step > 0) {  // every thread keeps its column sf_j, rows sf_r0, +sf_step, ...
          for (int r = sf_r0; r < n; r += sf_step)
            p.recv_sf[(int64_t)meta[s].rows[r] * nb + sf_j] = sf[sf_j];
        } else {
          for (int e = ctid; e < n * nb; e += nct) {
            const int r = e / nb, j = e - r * nb;
            p.recv_sf[(int64_t)meta[s].rows[r] * nb + j] = sf[j];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    } else {
      // BF16 or pre-quantised: the input stage is the payload; it is released
      // once its bulk stores have read it.
      if (!waited) {
        griddep_wait();
        waited = true;
      }
      if (!wait_or_fail(&rows[s])) return;
      const int n = meta[s].n;
      if (ctid == 0) {
        for (int r = 0; r < n; ++r)
          bulk_store_s2g_hint(recv + (int64_t)meta[s].rows[r] * out_bytes, in, (uint32_t)out_bytes,
                              stream_pol);
        bulk_commit();
        bulk_wait_read<0>();
      }
      if constexpr (MODE == kModePreq && !COL_MAJOR) {
        // row-major scales: the token's nb scales to each of its rows
        for (int e = ctid; e < n * nb; e += nct) {
          const int r = e / nb, j = e - r * nb;
          p.recv_sf[(int64_t)meta[s].rows[r] * nb + j] =
              __ldg(p.xs + (int64_t)t * p.xs_ts + (int64_t)j * p.xs_hs);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  if (!waited) griddep_wait();  // a CTA without tokens
  const bool pad_work = p.do_expand && (p.zero_padding || p.recv_w != nullptr);
  const int npad = pad_work ? __ldg(p.psum_pad + p.E) : 0;
  const int64_t pad_items = (npad + kPadRowsPerItem - 1) / kPadRowsPerItem;
  // The CTA's tokens are done: publish that their per-token scales are
  // written and let the scale gather launch.  Then the padding items.
  if constexpr (FP8 && COL_MAJOR) {
    if (p.sf_wait == kSfWaitHandshake) {
      __threadfence();
      named_barrier(kBarConsumers, nct);
      if (ctid == 0) atomicAdd(p.sf_sync, 1);
    }
  }
  griddep_launch_dependents();
  // Padding items, also handed out dynamically; the next index is fetched
  // while the current item is written.
  __shared__ int pad_item_s[2];
  int next_item = 0;
  if (ctid == 0 && pad_items > 0) next_item = atomicAdd(p.sched + 2, 1);
  for (int pi = 0; pad_items > 0; ++pi) {
    if (ctid == 0) pad_item_s[pi & 1] = next_item;
    named_barrier(kBarConsumers, nct);
    const int item = pad_item_s[pi & 1];
    if (item >= pad_items) break;
    if (ctid == 0) next_item = atomicAdd(p.sched + 2, 1);
    zero_padding_item(p, item, npad, prow_s[pi & 1], FP8_OUT, COL_MAJOR, ctid, nct);
  }
  if (ctid == 0) {
    bulk_wait_all<0>();
    // the last CTA resets the scheduler for the next dispatch on the handle
    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      p.sched[0] = 0;
      p.sched[1] = 0;
      p.sched[2] = 0;
    }
  }
}

// Column-major scale factors of every destination row, gathered from the
// per-token scales (sf_src: the dispatch kernel's own, or the caller's for a
// pre-quantised input) through the row's source token (recv_src_metadata).
// One work item (row, g) loads 16 bytes of its token's scales and writes
// scale blocks 4g..4g+3 of its row; the threads of a warp take 32
// consecutive rows of one g, so every store of a warp is contiguous.
// Padding rows get 0.
__device__ __forceinline__ void sf_expand_one(const DispatchParams &p, int nb, int j0, int tok,
                                              float *dst) {
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (tok >= 0) {
    // scales written by the running dispatch kernel are read through L2 only
    const float *src = p.sf_src + (int64_t)tok * p.sf_src_ts + (int64_t)j0 * p.sf_src_hs;
    if (p.sf_src_vec4) {
      const float4 q = p.sf_wait == kSfWaitHandshake ? __ldcg(reinterpret_cast<const float4 *>(src))
                                 : __ldg(reinterpret_cast<const float4 *>(src));
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      for (int u = 0; u < 4 && j0 + u < nb; ++u)
        v[u] = p.sf_wait == kSfWaitHandshake ? __ldcg(src + (int64_t)u * p.sf_src_hs)
                         : __ldg(src + (int64_t)u * p.sf_src_hs);
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (j0 + u < nb) dst[(int64_t)u * p.sf_hidden_stride] = v[u];
}

template <bool FIXED>
__device__ __forceinline__ void sf_expand_body(const DispatchParams &p) {
  const int nb = p.H / kFp8Block;
  const int2 *meta = reinterpret_cast<const int2 *>(p.meta);
  if constexpr (FIXED) {
    // grid (x, 1, E): the CTAs of expert e walk its used rows i < count,
    // group of 4 scale blocks by group, consecutive threads on consecutive
    // rows of one group (coalesced stores into the expert's column-major slab)
    const int e = blockIdx.z;
    const int64_t n = min((int64_t)__ldg(p.cnt_e + e), (int64_t)p.fixed_cap);
    const int64_t items = n * ((nb + 3) / 4);
    const int64_t row0 = (int64_t)e * p.fixed_cap;
    float *out0 = p.recv_sf + (int64_t)e * p.sf_expert_stride;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * blockDim.x) {
      const int64_t g = it / n, i = it - g * n;
      const int j0 = (int)g * 4;
      sf_expand_one(p, nb, j0, __ldg(&meta[row0 + i].x),
                    out0 + i + (int64_t)j0 * p.sf_hidden_stride);
    }
  } else {
    // one global column-major matrix over the rows below the layout's total:
    // grid (blocks of kSfRowsPerThread * 256 rows, groups of 4 scale blocks);
    // a thread takes rows r, r + 256, ... so each step of a warp stays
    // coalesced, and its kSfRowsPerThread metadata loads are all in flight
    const int64_t n = min((int64_t)__ldg(p.num_rows), p.rows_alloc);
    const int64_t row0 = (int64_t)blockIdx.x * blockDim.x * kSfRowsPerThread + threadIdx.x;
    const int j0 = blockIdx.y * 4;
    int tok[kSfRowsPerThread];
#pragma unroll
    for (int u = 0; u < kSfRowsPerThread; ++u) {
      const int64_t row = row0 + (int64_t)u * blockDim.x;
      tok[u] = row < n ? __ldg(&meta[row].x) : -2;
    }
#pragma unroll
    for (int u = 0; u < kSfRowsPerThread; ++u) {
      const int64_t row = row0 + (int64_t)u * blockDim.x;
      if (tok[u] != -2)
        sf_expand_one(p, nb, j0, tok[u], p.recv_sf + row + (int64_t)j0 * p.sf_hidden_stride);
    }
  }
}

template <bool FIXED>
__global__ void __launch_bounds__(256) sf_expand_kernel(DispatchParams p) {
  // Launched while the dispatch kernel still runs (programmatic dependent
  // launch).  With sf_wait the per-token scales come from that kernel: wait,
  // bounded, until every dispatch CTA has published its tokens' scales.
  // The next kernel may start its own prologue at once.
  if (p.sf_wait == kSfWaitGrid) griddep_wait();
  griddep_launch_dependents();
  __shared__ int ready;
  if (threadIdx.x == 0) {
    bool ok = true;
    if (p.sf_wait == kSfWaitHandshake) {
      ok = false;
      for (int it = 0; it < kSfWaitIters && !ok; ++it) {
        ok = ld_acquire_gpu(p.sf_sync) >= p.sf_sync_target;
        if (!ok) __nanosleep(256);
      }
      if (!ok) atomicOr(p.err, EP_ERRBIT_TIMEOUT);
    }
    ready = ok;
  }
  __syncthreads();
  if (ready) sf_expand_body<FIXED>(p);
  if (p.sf_wait == kSfWaitHandshake) {
    // the last CTA resets the handshake for the next dispatch on this handle
    __syncthreads();
    if (threadIdx.x == 0) {
      const int total = (int)(gridDim.x * gridDim.y * gridDim.z);
      if (atomicAdd(p.sf_sync + 1, 1) == total - 1) {
        p.sf_sync[0] = 0;
        p.sf_sync[1] = 0;
      }
    }
  }
  // This kernel ends only after the dispatch kernel has: a kernel launched
  // after it with programmatic dependent launch waits for this one alone.
  if (p.sf_wait != kSfWaitGrid) griddep_wait();
}

template <int MODE, bool CM>
cudaError_t launch_one(const DispatchParams &p0, int sm_cap, cudaStream_t s) {
  constexpr bool FP8 = MODE == kModeQuant;
  DispatchParams p = p0;
  // the scale gather reads 4 scales of a token at once when they are
  // contiguous and 16-byte aligned
  p.sf_src_vec4 = (p.H / kFp8Block) % 4 == 0 && p.sf_src_hs == 1 && p.sf_src_ts % 4 == 0 &&
                  reinterpret_cast<uintptr_t>(p.sf_src) % 16 == 0;
  const int H = p.H;
  const int nvec = H / 8;
  // FP8: consumer threads cover the row in whole 16-lane groups; BF16: the
  // consumers only issue bulk copies and zero padding rows.
  const int consumers = FP8 ? std::min(kMaxConsumers, (nvec + 31) / 32 * 32) : 64;
  const int threads = consumers + 32;
  const size_t in_stage = (size_t)((MODE == kModePreq ? H : 2 * H) + 127) / 128 * 128;
  const size_t out_stage = FP8 ? (size_t)(H + 127) / 128 * 128 : 0;
  const size_t sf_stage = FP8 && !CM ? sizeof(float) * ((H / kFp8Block + 31) / 32 * 32) : 0;
  // Two stages for quantised rows of the largest hidden sizes (above ~24K:
  // three do not fit), and for quantising up to kFewTokens tokens: a CTA
  // then holds few tokens, the quantisation is bound by instruction latency,
  // and the smaller ring lets 5 CTAs share an SM instead of 3 (measured:
  // prefill 69.8 -> 68.7 us, decode 18.0 -> 17.2 us, decode_ll step 54.9 ->
  // 52.8 us).  Copies and long batches keep three (two stages: large 388.7 ->
  // 402.0 us, the BF16 skewed dispatch 85.0 -> 86.9 us).
  auto kern = dispatch_kernel<MODE, CM, kStages>;
  int stages = kStages;
  if constexpr (FP8) {
    if (kStages * (in_stage + out_stage + sf_stage) > kSmemLimit || p.T <= kFewTokens) {
      kern = dispatch_kernel<MODE, CM, 2>;
      stages = 2;
    }
  }
  const size_t smem = stages * (in_stage + out_stage + sf_stage);
  int dev = 0, per_sm = 0;
  cudaError_t err =
      launch_geometry(reinterpret_cast<const void *>(kern), threads, smem, &dev, &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int sms = device_sm_count(dev);
  const int use_sms = (sm_cap > 0 && sm_cap < sms) ? sm_cap : sms;
  const int64_t items = (int64_t)p.T + p.max_pad_items;
  const int64_t grid = std::min<int64_t>((int64_t)use_sms * per_sm, items);
  if (grid <= 0) return cudaSuccess;
  p.sf_sync_target = (int)grid;        // every dispatch CTA publishes once
  // quantising: the gather needs the kernel's scales -- by the handshake, or
  // (fixed capacity: few rows per expert) after the whole kernel
  p.sf_wait = MODE != kModeQuant ? kSfWaitNone
              : p.fixed_cap > 0  ? kSfWaitGrid
                                 : kSfWaitHandshake;
  {
    // programmatic dependent launch: the prologue overlaps the previous kernel
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3(threads);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    err = cudaLaunchKernelEx(&lc, kern, p);
  }
  if (err != cudaSuccess || MODE == kModeBf16 || !CM) return err;
  // column-major scales: one gather pass (rows past the real total, in an
  // upper-bound allocation, are left untouched; so are the unused rows of a
  // fixed-capacity slab)
  const int groups = (H / kFp8Block + 3) / 4;
  dim3 sf_grid;
  if (p.fixed_cap > 0)  // per expert: up to 4 CTAs striding over its (row, group) items
    sf_grid = dim3((unsigned)std::min<int64_t>(4, ((int64_t)p.fixed_cap * groups + 2047) / 2048), 1,
                   (unsigned)p.E);
  else
    sf_grid = dim3((unsigned)((p.rows_alloc + 256 * kSfRowsPerThread - 1) / (256 * kSfRowsPerThread)),
                   (unsigned)groups);
  if (p.rows_alloc > 0) {
    // launched as soon as every dispatch CTA is past its tokens
    cudaLaunchConfig_t lc{};
    lc.gridDim = sf_grid;
    lc.blockDim = dim3(256);
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    err = p.fixed_cap > 0 ? cudaLaunchKernelEx(&lc, sf_expand_kernel<true>, p)
                         : cudaLaunchKernelEx(&lc, sf_expand_kernel<false>, p);
  }
  return err;
}

}  // namespace

cudaError_t launch_dispatch(const DispatchParams &p, int mode, int col_major, int sm_cap,
                            cudaStream_t s) {
  if (mode == kModeQuant)
    return col_major ? launch_one<kModeQuant, true>(p, sm_cap, s)
                     : launch_one<kModeQuant, false>(p, sm_cap, s);
  if (mode == kModePreq)
    return col_major ? launch_one<kModePreq, true>(p, sm_cap, s)
                     : launch_one<kModePreq, false>(p, sm_cap, s);
  return launch_one<kModeBf16, false>(p, sm_cap, s);
}

}  // namespace ep
