// Combine: per-token weighted gather-reduce of expert outputs, fp32 -> BF16.
//
// Follows "DeepEP V2 notes, ch. 8: combine, handle and async overlap", §8.1
// (combine walks the dispatch handle backwards, with optional bias and top-k
// weights) and the vLLM PR #52781 review (combine takes BF16 expert output;
// with topk_weights = None the caller has already applied the weights).
//
// Work unit = (token, chunk of the hidden dimension).  Persistent CTAs, warp
// specialised:
//   warp 0 (producer) reads a unit's routing (destination rows, weights,
//     expert ids; prefetched four units ahead), compacts the valid slots
//     (dropping repeated rows when there are no weights) and issues one
//     cp.async.bulk global->shared copy per slot row chunk (plus the per-token
//     bias chunks) into a ring of kStages shared-memory stages, completion
//     counted on the stage's "full" mbarrier;
//   the other warps (consumers) wait for a stage and accumulate its rows
//     strictly in slot order, each thread one 16-byte vector of the chunk
//     (with a per-expert bias) or two (otherwise): the per-expert bias added
//     to each row first (a small table reused by every token: read through
//     L1, not staged; one mixed-precision BF16 + fp32 add per element), then
//     separately rounded fp32 multiplies and adds (__fmul_rn / __fadd_rn:
//     never contracted to an FMA); then the per-token biases are added, the
//     sums rounded to BF16 (nearest even) and stored, and the stage released
//     on its "empty" mbarrier.
// Each output element is written by exactly one thread: no atomics.  Every
// mbarrier wait is bounded; a wait that gives up sets EP_ERRBIT_TIMEOUT in
// the handle's error word and the CTA returns.
#include <algorithm>

#include "ep_internal.cuh"
#include "ep_ptx.cuh"

namespace ep {
namespace {

constexpr int kStages = 3;
constexpr int kMaxConsumers = 224;
constexpr int64_t kStageBudget = 96 * 1024;    // shared-memory stages per CTA
constexpr int64_t kEbStageBudget = 48 * 1024;  // same, with a per-expert bias
constexpr int kWaitIters = 4000;          // x kWaitHintNs: gives up after ~2 s
constexpr uint32_t kWaitHintNs = 500000;

struct __align__(8) SlotMeta {
  float w;
  int e;
};

struct StageMeta {
  SlotMeta m[EP_MAX_TOPK];  // weight and expert of each valid slot: one 8-byte read
  int n;                    // valid slots in this unit
};

__device__ __forceinline__ void unpack8(const uint4 &v, float *f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

struct Routing {
  int d, e;
  float w;
};

template <bool HAS_W, bool HAS_EB>
__device__ __forceinline__ Routing load_routing(const CombineParams &p, int64_t t, int lane) {
  Routing r{-1, -1, 1.f};
  if (lane < p.K) {
    r.d = __ldg(p.dst + t * p.K + lane);
    if (HAS_EB) r.e = __ldg(p.topk32 + t * p.K + lane);
    if (HAS_W) r.w = __ldg(p.topk_w + t * p.K + lane);
  }
  return r;
}

// A CTA's current unit u and its (token t, chunk c), advanced by the grid
// stride G.  STEP: with adds only (gq whole tokens and gr chunks per stride);
// otherwise t and c are recomputed from u by a 64-bit division.
template <bool STEP>
struct UnitCursor {
  int64_t u;
  int t, c;
  __device__ __forceinline__ UnitCursor(int64_t u0, int nchunks)
      : u(u0), t((int)(u0 / nchunks)), c((int)(u0 % nchunks)) {}
  __device__ __forceinline__ void advance(int64_t G, int gq, int gr, int nchunks) {
    u += G;
    if (STEP) {
      t += gq;
      c += gr;
      if (c >= nchunks) {
        c -= nchunks;
        ++t;
      }
    } else {
      t = (int)(u / nchunks);
      c = (int)(u - (int64_t)t * nchunks);
    }
  }
};

// One consumer thread's share of a unit: NV vectors, vstep vectors apart,
// each reduced over the unit's slots in slot order.
template <int NV, bool HAS_W, bool HAS_EB>
__device__ __forceinline__ void reduce_vectors(const CombineParams &p, const StageMeta &m,
                                               const uint8_t *sb, int chunk_bytes, int v,
                                               int vstep, int64_t off, int64_t t, int nbias) {
  const int H = p.H;
  const int64_t row_bytes = 2 * (int64_t)H;
  const int n = m.n;
  float acc[NV][8];
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[k][q] = 0.f;
  const uint16_t *eb_v = HAS_EB ? p.ebias + off / 2 + v * 8 : nullptr;  // this vector's bias
  for (int j = 0; j < n; ++j) {
    const SlotMeta sm = m.m[j];
    const uint8_t *yp = sb + (uint32_t)(j * chunk_bytes + v * 16);
    const uint16_t *eb_e = HAS_EB ? eb_v + (int64_t)sm.e * H : nullptr;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float f[8];
      const uint4 yv = *reinterpret_cast<const uint4 *>(yp + (uint32_t)(k * vstep * 16));
      if (HAS_EB) {
        // y + expert bias: one mixed-precision add per element, y taken as
        // BF16 straight from its half-word, the bias widened to fp32
        const uint4 bv = ld_cached_v4(eb_e + k * vstep * 8);
        add2_bf16_f32(yv.x, bf16_lo(bv.x), bf16_hi(bv.x), f[0], f[1]);
        add2_bf16_f32(yv.y, bf16_lo(bv.y), bf16_hi(bv.y), f[2], f[3]);
        add2_bf16_f32(yv.z, bf16_lo(bv.z), bf16_hi(bv.z), f[4], f[5]);
        add2_bf16_f32(yv.w, bf16_lo(bv.w), bf16_hi(bv.w), f[6], f[7]);
      } else {
        unpack8(yv, f);
      }
      if (HAS_W) {
        const float w = sm.w;
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[k][q] = __fadd_rn(acc[k][q], __fmul_rn(w, f[q]));
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[k][q] = __fadd_rn(acc[k][q], f[q]);
      }
    }
  }
  for (int b = 0; b < nbias; ++b) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4 *>(
                  sb + (uint32_t)((n + b) * chunk_bytes + (v + k * vstep) * 16)),
              f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[k][q] = __fadd_rn(acc[k][q], f[q]);
    }
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    uint4 o;
    o.x = cvt_bf16x2(acc[k][0], acc[k][1]);
    o.y = cvt_bf16x2(acc[k][2], acc[k][3]);
    o.z = cvt_bf16x2(acc[k][4], acc[k][5]);
    o.w = cvt_bf16x2(acc[k][6], acc[k][7]);
    st_stream_v4(reinterpret_cast<uint8_t *>(p.out) + t * row_bytes + off +
                     (int64_t)(v + k * vstep) * 16,
                 o);
  }
}

template <bool HAS_W, bool HAS_EB, int NV, bool STEP>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1)
    combine_kernel(CombineParams p, int chunk_bytes, int nchunks, int slots_cap) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t empty[kStages];
  __shared__ StageMeta meta[kStages];

  const int H = p.H;
  const int64_t row_bytes = 2 * (int64_t)H;
  const int64_t stage_bytes = (int64_t)slots_cap * chunk_bytes;
  // STEP: units stepped with adds only (the launcher's choice).
  using Cursor = UnitCursor<STEP>;
  const int64_t G = gridDim.x;
  const int gq = (int)(G / nchunks), gr = (int)(G % nchunks);
  const int has_b0 = p.bias0 != nullptr, has_b1 = p.bias1 != nullptr;
  const int nbias = has_b0 + has_b1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncw = (blockDim.x >> 5) - 1;  // consumer warps

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // Launched with programmatic dependent launch: the set-up above overlaps
  // the tail of the kernel before this one; nothing below touches global
  // memory before that kernel's writes are visible.
  griddep_wait();

  if (warp == 0) {
    // ---------------- producer ----------------
    const uint64_t stream_pol = l2_policy_evict_first();  // expert outputs are read once
    // routing of the next four units is in flight while one is issued
    // (ahead: the unit whose routing was loaded last)
    Cursor u(blockIdx.x, nchunks), ahead(blockIdx.x, nchunks);
    Routing r0{-1, -1, 1.f}, r1{-1, -1, 1.f}, r2{-1, -1, 1.f}, r3{-1, -1, 1.f};
    if (ahead.t < p.T) r0 = load_routing<HAS_W, HAS_EB>(p, ahead.t, lane);
    ahead.advance(G, gq, gr, nchunks);
    if (ahead.t < p.T) r1 = load_routing<HAS_W, HAS_EB>(p, ahead.t, lane);
    ahead.advance(G, gq, gr, nchunks);
    if (ahead.t < p.T) r2 = load_routing<HAS_W, HAS_EB>(p, ahead.t, lane);
    ahead.advance(G, gq, gr, nchunks);
    if (ahead.t < p.T) r3 = load_routing<HAS_W, HAS_EB>(p, ahead.t, lane);
    for (int64_t i = 0; u.t < p.T; ++i, u.advance(G, gq, gr, nchunks)) {
      const Routing cur = r0;
      r0 = r1;
      r1 = r2;
      r2 = r3;
      ahead.advance(G, gq, gr, nchunks);
      if (ahead.t < p.T) r3 = load_routing<HAS_W, HAS_EB>(p, ahead.t, lane);
      const int s = (int)(i % kStages);
      const int64_t k = i / kStages;
      if (k > 0) {
        bool ok = false;
        if (lane == 0) ok = mbar_wait_bounded(&empty[s], (uint32_t)((k - 1) & 1), kWaitIters,
                                              kWaitHintNs);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) atomicOr(p.err, EP_ERRBIT_TIMEOUT);
          return;
        }
      }
      const int64_t t = u.t;
      const int64_t off = (int64_t)u.c * chunk_bytes;
      const uint32_t bytes = (uint32_t)min((int64_t)chunk_bytes, row_bytes - off);
      bool use = cur.d >= 0;
      if (!HAS_W) {  // weights already applied: each row counts once
        const unsigned peers = __match_any_sync(0xffffffffu, cur.d);
        use = use && lane == __ffs(peers) - 1;
      }
      const unsigned m = __ballot_sync(0xffffffffu, use);
      const int n = __popc(m);
      const int pos = __popc(m & lanemask_lt());
      if (use) {
        meta[s].m[pos] = SlotMeta{cur.w, cur.e};
      }
      if (lane == 0) meta[s].n = n;
      __syncwarp();
      const int rows = n + has_b0 + has_b1;
      if (lane == 0) {
        if (rows > 0)
          mbar_arrive_expect_tx(&full[s], (uint32_t)rows * bytes);
        else
          mbar_arrive(&full[s]);
      }
      __syncwarp();
      uint8_t *sb = smem + s * stage_bytes;
      if (use) {
        bulk_load_g2s_hint(sb + (int64_t)pos * chunk_bytes,
                           reinterpret_cast<const uint8_t *>(p.y) + (int64_t)cur.d * row_bytes + off,
                           bytes, &full[s], stream_pol);
      }
      const int brow = n;
      if (lane == 0 && has_b0)
        bulk_load_g2s(sb + (int64_t)brow * chunk_bytes,
                      reinterpret_cast<const uint8_t *>(p.bias0) + t * row_bytes + off, bytes,
                      &full[s]);
      if (lane == 1 && has_b1)
        bulk_load_g2s(sb + (int64_t)(brow + has_b0) * chunk_bytes,
                      reinterpret_cast<const uint8_t *>(p.bias1) + t * row_bytes + off, bytes,
                      &full[s]);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = threadIdx.x - 32;
  const int cthreads = blockDim.x - 32;
  int64_t i = 0;
  for (Cursor u(blockIdx.x, nchunks); u.t < p.T; u.advance(G, gq, gr, nchunks), ++i) {
    const int s = (int)(i % kStages);
    const uint32_t par = (uint32_t)((i / kStages) & 1);
    if (!mbar_wait_bounded(&full[s], par, kWaitIters, kWaitHintNs)) {
      if (lane == 0) atomicOr(p.err, EP_ERRBIT_TIMEOUT);
      return;
    }
    const int64_t t = u.t;
    const int64_t off = (int64_t)u.c * chunk_bytes;
    const int nv = (int)(min((int64_t)chunk_bytes, row_bytes - off) / 16);
    const uint8_t *sb = smem + (uint32_t)(s * (int)stage_bytes);
    for (int v = ctid; v < nv; v += NV * cthreads) {
      if (NV == 2 && v + cthreads < nv)
        reduce_vectors<2, HAS_W, HAS_EB>(p, meta[s], sb, chunk_bytes, v, cthreads, off, t, nbias);
      else
        reduce_vectors<1, HAS_W, HAS_EB>(p, meta[s], sb, chunk_bytes, v, cthreads, off, t, nbias);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// Units per CTA up to which the units are stepped with adds only.
constexpr int64_t kStepUnitsPerCta = 16;

template <bool W, bool EB, int NV>
cudaError_t launch_one(const CombineParams &p, int sm_cap, cudaStream_t s) {
  const int64_t row_bytes = 2 * (int64_t)p.H;
  const int nbias = (p.bias0 != nullptr) + (p.bias1 != nullptr);
  const int slots_cap = p.K + nbias;
  // Stage budget ~96 KB per CTA (two CTAs per SM).  With a per-expert bias
  // half of it: the bias rows are read through L1, which keeps what shared
  // memory leaves free.  Chunks are equal-sized multiples of 512 bytes where
  // the row allows (whole L2 lines for the bias reads), else of 16 bytes.
  const int64_t budget = (EB ? kEbStageBudget : kStageBudget) / kStages;
  const int64_t gran = row_bytes >= 512 ? 512 : 16;
  int64_t chunk = std::max<int64_t>(gran, budget / slots_cap / gran * gran);
  chunk = std::min(chunk, row_bytes);
  const int64_t n0 = (row_bytes + chunk - 1) / chunk;
  chunk = std::min(row_bytes, ((row_bytes + n0 - 1) / n0 + gran - 1) / gran * gran);
  chunk = (chunk + 15) / 16 * 16;
  const int nchunks = (int)((row_bytes + chunk - 1) / chunk);  // every chunk non-empty
  const int nv = (int)(chunk / 16);
  const int consumers = std::min(kMaxConsumers, ((nv + NV - 1) / NV + 31) / 32 * 32);
  const int threads = consumers + 32;
  const size_t smem = (size_t)kStages * slots_cap * chunk;
  const int64_t units = (int64_t)p.T * nchunks;
  // Unit cursor: adds only for the expert-bias combine (bound by instruction
  // issue: skewed 162 -> 152 us) and for short combines, where each CTA's
  // 64-bit divisions lie on its latency path (decode 23.3 -> 21.1 us, step
  // 39.9 -> 38.0 us); the long HBM-bound combines measured faster with the
  // division (prefill 78.3 -> 76.2 us, 32768 tokens 635 -> 624 us).  The
  // grid, and so the choice, comes from the stepping kernel's occupancy; the
  // division kernel has its own shared-memory opt-in and occupancy.
  auto kern = combine_kernel<W, EB, NV, true>;
  const void *func = reinterpret_cast<const void *>(kern);
  int dev = 0, per_sm = 0;
  cudaError_t err = launch_geometry(func, threads, smem, &dev, &per_sm);
  if (err != cudaSuccess) return err;
  const int sms = device_sm_count(dev);
  const int use_sms = (sm_cap > 0 && sm_cap < sms) ? sm_cap : sms;
  int64_t grid = std::min<int64_t>((int64_t)use_sms * std::max(per_sm, 1), units);
  if constexpr (!EB) {
    if (units > kStepUnitsPerCta * grid) {
      kern = combine_kernel<W, EB, NV, false>;
      func = reinterpret_cast<const void *>(kern);
      err = launch_geometry(func, threads, smem, &dev, &per_sm);
      if (err != cudaSuccess) return err;
      grid = std::min<int64_t>((int64_t)use_sms * std::max(per_sm, 1), units);
    }
  }
  if (grid <= 0) return cudaSuccess;
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
  return cudaLaunchKernelEx(&lc, kern, p, (int)chunk, nchunks, slots_cap);
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, int sm_cap, cudaStream_t s) {
  const bool w = p.topk_w != nullptr, eb = p.ebias != nullptr;
  // Vectors per consumer thread: two halve the per-unit consumer warps and
  // give each slot two independent loads (decode combine 25.2 -> 23.3 us);
  // with a per-expert bias the second vector's bias reads made the
  // issue-bound reduction slower (skewed 136 -> 158 us), so it keeps one.
  if (w && eb) return launch_one<true, true, 1>(p, sm_cap, s);
  if (w) return launch_one<true, false, 2>(p, sm_cap, s);
  if (eb) return launch_one<false, true, 1>(p, sm_cap, s);
  return launch_one<false, false, 2>(p, sm_cap, s);
}

}  // namespace ep
