// Routing layout: counts, prefix sums, destination rows and source metadata.
//
// Follows the layout contract of "DeepEP V2 notes, ch. 7: how V2 dispatch
// builds expert inputs" (§7.2 layout metadata, §7.4 expanded layout) and the
// get_dispatch_layout outputs of the DeepEP README interface example.
//
// Tokens are cut into chunks of up to kLayoutChunkTokens tokens that never
// straddle a source rank; one CTA owns one chunk in both kernels (256 threads,
// one per token, in count; 1024 in assign).
//   count  - one thread per token: validates and copies topk_idx, builds the
//            token's rank set (is_token_in_rank, first slot per rank) and
//            adds to the CTA's expert / rank histograms, stored block-major.
//   assign - every CTA sums the histogram columns it needs (global totals
//            and the totals of the chunks before it), scans them into segment
//            starts, then ranks its own slots stably: warps walk contiguous
//            runs of (token, slot) pairs in order, ranking equal keys with
//            shared 64-bit words (a running count plus the mask of the lanes
//            holding the key in the current step).  Row = segment start +
//            earlier chunks +
//            earlier warps + earlier lanes, i.e. ascending (token, slot)
//            inside every segment, with no atomics deciding positions.  One
//            extra CTA, which owns no chunk, writes the global counts and
//            prefix sums (and, for the host count wait, the mapped totals).
#include <algorithm>

#include "ep_internal.cuh"
#include "ep_ptx.cuh"

namespace ep {
namespace {

constexpr int NT = kLayoutThreads;     // assign kernel: 1024 threads
constexpr int NWARPS = NT / 32;
constexpr int NTC = kLayoutChunkTokens;  // count kernel: one thread per token

__device__ __forceinline__ int chunk_of(const LayoutParams &p, int b, int &t0) {
  const int s = b / p.blocks_per_src;
  const int c = b - s * p.blocks_per_src;
  const int64_t start = (int64_t)s * p.M + (int64_t)c * p.chunk_tokens;
  const int64_t src_end = min((int64_t)(s + 1) * p.M, (int64_t)p.T);
  const int64_t end = min(start + p.chunk_tokens, src_end);
  t0 = (int)min(start, (int64_t)p.T);
  return end > start ? (int)(end - start) : 0;
}

// Exclusive scan of f(i), i < n, by the whole CTA into out[0..n]; returns the
// total.  `warp_tot` is shared scratch of NWARPS + 1 ints.
template <typename F>
__device__ int cta_exclusive_scan(int n, F f, int32_t *out, int *warp_tot) {
  const int per = (n + NT - 1) / NT;
  const int beg = min(threadIdx.x * per, n);
  const int end = min(beg + per, n);
  int local = 0;
  for (int i = beg; i < end; ++i) local += f(i);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NWARPS ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    if (lane < NWARPS) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == NWARPS - 1) warp_tot[NWARPS] = wi;
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - local;
  for (int i = beg; i < end; ++i) {
    out[i] = run;
    run += f(i);
  }
  const int total = warp_tot[NWARPS];
  if (threadIdx.x == 0) out[n] = total;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(NTC) layout_count_kernel(LayoutParams p) {
  extern __shared__ __align__(16) int smem[];
  const int K = p.K, L = p.L, R = p.R, E = p.E;
  int *hist_e = smem;                       // [E]
  int *hist_r = hist_e + E;                 // [R]
  int *rank_of = hist_r + R;                // [E] owning rank of each expert
  int *idx_s = rank_of + E;                 // [chunk_tokens * K]
  __shared__ unsigned err_s;
  const int b = blockIdx.x;
  int t0;
  const int nt = chunk_of(p, b, t0);
  const int ns = nt * K;
  const int64_t base = (int64_t)t0 * K;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) err_s = 0;
  for (int i = threadIdx.x; i < E + R; i += NTC) smem[i] = 0;
  for (int e = threadIdx.x; e < E; e += NTC) rank_of[e] = e / L;

  // Coalesced load of the chunk, eight loads in flight per thread: validate
  // and keep an int32 copy.
  unsigned err = 0;
  constexpr int kBatch = 8;
  for (int i0 = threadIdx.x; i0 < ns; i0 += NTC * kBatch) {
    long long v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * NTC;
      v[u] = -1;
      if (i < ns)
        v[u] = p.idx_is_int64 ? __ldg(static_cast<const long long *>(p.topk_idx) + base + i)
                              : __ldg(static_cast<const int *>(p.topk_idx) + base + i);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * NTC;
      if (i >= ns) break;
      long long x = v[u];
      if (x < -1 || x >= E) {
        err |= EP_ERRBIT_BAD_TOPK_IDX;
        x = -1;
      }
      idx_s[i] = static_cast<int>(x);
      p.topk32[base + i] = static_cast<int>(x);
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  __syncthreads();
  griddep_launch_dependents();  // the assign kernel's prologue may start now
  if (lane == 0 && err) atomicOr(&err_s, err);

  // One thread per token: expert histogram and the token's rank set.
  const int tl = threadIdx.x;
  const bool active = tl < nt;
  const int *trow = idx_s + tl * K;
  uint64_t mask = 0;  // rank set (R <= 64)
  if (active) {
    for (int k = 0; k < K; ++k) {
      const int e = trow[k];
      if (e < 0) continue;
      atomicAdd(&hist_e[e], 1);
      const int r = rank_of[e];
      if (R <= 64) {
        mask |= 1ull << r;
      } else {
        bool first = true;  // wide rank sets: look back at this token's slots
        for (int j = 0; j < k && first; ++j) first = !(trow[j] >= 0 && rank_of[trow[j]] == r);
        if (first) atomicAdd(&hist_r[r], 1);
      }
    }
  }
  if (R <= 32) {
    for (int r = 0; r < R; ++r) {
      const int c = __popc(__ballot_sync(0xffffffffu, (mask >> r) & 1));
      if (lane == 0 && c) atomicAdd(&hist_r[r], c);
    }
  } else if (R <= 64) {
    for (uint64_t m = mask; m; m &= m - 1) atomicAdd(&hist_r[__ffsll((long long)m) - 1], 1);
  }
  if (active) {
    uint8_t *row = p.in_rank + ((int64_t)t0 + tl) * R;
    if (R <= 64) {
      if ((R & 3) == 0) {
        for (int r = 0; r < R; r += 4) {
          const uint32_t w = (uint32_t)((mask >> r) & 1) | (uint32_t)((mask >> (r + 1)) & 1) << 8 |
                             (uint32_t)((mask >> (r + 2)) & 1) << 16 |
                             (uint32_t)((mask >> (r + 3)) & 1) << 24;
          *reinterpret_cast<uint32_t *>(row + r) = w;
        }
      } else {
        for (int r = 0; r < R; ++r) row[r] = (uint8_t)((mask >> r) & 1);
      }
    } else {
      for (int r = 0; r < R; ++r) row[r] = 0;
      for (int k = 0; k < K; ++k)
        if (trow[k] >= 0) row[rank_of[trow[k]]] = 1;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += NTC) p.blk_e[(int64_t)b * E + e] = hist_e[e];
  for (int r = threadIdx.x; r < R; r += NTC) p.blk_r[(int64_t)b * R + r] = hist_r[r];
  if (threadIdx.x == 0) p.blk_err[b] = err_s;
}

__global__ void __launch_bounds__(NT, 1) layout_assign_kernel(LayoutParams p) {
  extern __shared__ __align__(16) int smem[];
  const int K = p.K, L = p.L, E = p.E, R = p.R, A = p.A;
  const int nkey = p.do_expand ? E : R;
  const int cap = p.chunk_tokens * K;
  int *idx_s = smem;                  // [cap]
  int *row_s = idx_s + cap;           // [cap] sort key, then row
  int *tot_s = row_s + cap;           // [E + R] global totals
  int *bef_s = tot_s + E + R;         // [E + R] totals of the chunks before this one
  int *seg_s = bef_s + E + R;         // [nkey + 1] segment starts
  int *rank_of = seg_s + nkey + 1;    // [E] owning rank of each expert
  int *scan_s = rank_of + E;          // [2E + R + 1] outputs CTA: prefix sums
  // [rank_warps][nkey] 64-bit words: low half = running count of the key in
  // the warp's range, high half = lanes holding the key in the current step
  unsigned long long *whist =
      reinterpret_cast<unsigned long long *>(scan_s + 2 * E + R + 1 + ((nkey + E + R) & 1));
  __shared__ int warp_tot[NWARPS + 1];

  const int b = blockIdx.x;
  int t0;
  const int nt = chunk_of(p, b, t0);
  const int ns = nt * K;
  const int64_t base = (int64_t)t0 * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nrw = p.rank_warps;

  for (int i = threadIdx.x; i < nrw * nkey; i += NT) whist[i] = 0ull;
  for (int e = threadIdx.x; e < E; e += NT) rank_of[e] = e / L;
  griddep_wait();  // everything below reads the count kernel's outputs
  griddep_launch_dependents();  // the next kernel (dispatch) may start its prologue
  for (int i = threadIdx.x; i < ns; i += NT) idx_s[i] = p.topk32[base + i];
  // Column sums of the per-chunk histograms: global totals and this chunk's
  // offset.  g consecutive lanes share a key and split its chunks.
  {
    const int nk = E + R;
    int g = 1;
    while (g < 32 && g * 2 * nk <= NT) g <<= 1;
    const int sub = threadIdx.x & (g - 1);
    for (int key = threadIdx.x / g; key < nk + (NT / g - 1) - (nk + NT / g - 1) % (NT / g);
         key += NT / g) {
      int tot = 0, bef = 0;
      if (key < nk) {
        const int32_t *col = key < E ? p.blk_e + key : p.blk_r + (key - E);
        const int stride = key < E ? E : R;
        // batches of eight predicated loads, all in flight together
        for (int bb = sub; bb < p.num_blocks; bb += 8 * g) {
          int v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = bb + u * g;
            v[u] = c < p.num_blocks ? __ldcg(col + (int64_t)c * stride) : 0;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            tot += v[u];
            bef += (bb + u * g < b) ? v[u] : 0;
          }
        }
      }
      for (int o = g >> 1; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        bef += __shfl_xor_sync(0xffffffffu, bef, o);
      }
      if (key < nk && sub == 0) {
        tot_s[key] = tot;
        bef_s[key] = bef;
      }
    }
  }
  __syncthreads();

  // psum_rank_src[r][s], the tokens of source ranks < s that rank r
  // receives, is the rank total of the chunks before source rank s's first
  // chunk: that chunk's CTA holds it in bef_s.  Source ranks without tokens
  // (and s = R) get the full total, written by the outputs CTA.
  {
    const int RR = R + 1;
    const int src_real = p.T > 0 ? (int)(((int64_t)p.T + p.M - 1) / p.M) : 0;
    const int s = b / p.blocks_per_src;
    if (b == s * p.blocks_per_src && s < src_real)
      for (int r = threadIdx.x; r < R; r += NT) p.psum_rs[(int64_t)r * RR + s] = bef_s[E + r];
    if (b == p.num_blocks)
      for (int i = threadIdx.x; i < R * (RR - src_real); i += NT) {
        const int r = i / (RR - src_real), ss = src_real + (i - r * (RR - src_real));
        p.psum_rs[(int64_t)r * RR + ss] = tot_s[E + r];
      }
  }

  const int fcap = p.fixed_cap;
  if (b == p.num_blocks) {
    // Global outputs, written once by the extra CTA that owns no chunk (so no
    // ranking CTA waits for them).  One CTA-wide exclusive scan over
    // [counts | aligned counts | rank counts] gives every prefix sum (read
    // back by differences); then parallel stores, the totals and the host
    // notification.
    unsigned err = 0;
    if (warp == 0)  // issued before the scan, used after it
      for (int bb = lane; bb < p.num_blocks; bb += 32) err |= __ldcg(p.blk_err + bb);
    cta_exclusive_scan(
        2 * E + R,
        [&](int i) {
          return i < E ? tot_s[i] : i < 2 * E ? (tot_s[i - E] + A - 1) / A * A : tot_s[i - E];
        },
        scan_s, warp_tot);
    const int a0 = scan_s[E], r0 = scan_s[2 * E];
    for (int e = threadIdx.x; e <= E; e += NT) {
      const int pc = scan_s[e], pa = scan_s[E + e] - a0;
      if (e < E) {
        p.cnt_e[e] = tot_s[e];
        p.cnt_e_al[e] = (tot_s[e] + A - 1) / A * A;
      }
      p.psum_e[e] = fcap > 0 ? pc : pa;  // fixed capacity: the prefix of the counts
      p.psum_pad[e] = pa - pc;
    }
    for (int r = threadIdx.x; r <= R; r += NT) {
      if (r < R) p.cnt_r[r] = tot_s[E + r];
      p.psum_r[r] = scan_s[2 * E + r] - r0;
    }
    if (p.disp_sync != nullptr && threadIdx.x < kDispSyncWords) p.disp_sync[threadIdx.x] = 0;
    if (warp == 0) {
      err = __reduce_or_sync(0xffffffffu, err);
      bool over = false;
      if (fcap > 0)
        for (int e = lane; e < E; e += 32) over |= tot_s[e] > fcap;
      over = __any_sync(0xffffffffu, over);
      if (lane == 0) {
        const int num_recv = scan_s[2 * E + R] - r0;
        const int num_expanded = fcap > 0 ? a0 : r0 - a0;
        const int64_t total_rows = p.do_expand ? num_expanded : num_recv;
        if (fcap > 0 ? over : total_rows > p.row_limit) err |= EP_ERRBIT_OVERFLOW;
        p.ctrl[kCtrlError] = static_cast<int>(err);
        p.ctrl[kCtrlNumRecv] = num_recv;
        p.ctrl[kCtrlNumExpanded] = num_expanded;
        if (p.host != nullptr) {  // tagged words: no fence, the host checks each tag
          const uint64_t tag = (uint64_t)(uint32_t)p.seq << 32;
          p.host->num_recv = tag | (uint32_t)num_recv;
          p.host->num_expanded = tag | (uint32_t)num_expanded;
          p.host->error = tag | err;
        }
      }
    }
  } else if (fcap > 0) {
    // Segment starts of the sort key: the fixed per-expert capacity, the
    // aligned expert counts, or the rank counts.
    for (int e = threadIdx.x; e <= E; e += NT) seg_s[e] = e * fcap;
    __syncthreads();
  } else if (p.do_expand) {
    cta_exclusive_scan(E, [&](int e) { return (tot_s[e] + A - 1) / A * A; }, seg_s, warp_tot);
  } else {
    cta_exclusive_scan(R, [&](int r) { return tot_s[E + r]; }, seg_s, warp_tot);
  }
  if (b == p.num_blocks) return;  // the outputs CTA ranks nothing

  // Stable ranking: rank warp w owns the contiguous slot range [beg, end).
  // Pass 1 computes each slot's sort key -- the expert (expanded) or, for
  // the lowest slot of the token on each rank, the rank (rank layout) -- and
  // counts keys per warp (shared-memory atomics, order-free); after the
  // bases are known, pass 2 walks the range in order, 32 slots a step: every
  // lane ORs its bit into its key's word, the word then names the lanes
  // sharing the key (their order = slot order), and the lowest of them
  // advances the key's running count.  A word is two 32-bit halves (count,
  // lane mask), so both updates are 32-bit shared atomics and one 64-bit
  // load reads both.
  const int per_warp = (ns + nrw - 1) / nrw;
  const int beg = min(warp * per_warp, ns);
  const int end = warp < nrw ? min(beg + per_warp, ns) : beg;
  unsigned long long *wh = whist + (size_t)warp * nkey;
  for (int i = beg + lane; i < end; i += 32) {
    const int e = idx_s[i];
    int key = -1;
    if (e >= 0) {
      if (p.do_expand) {
        key = e;
      } else {
        const int tl = i / K, k = i - tl * K;
        const int r = rank_of[e];
        bool first = true;
        for (int j = 0; j < k && first; ++j) {
          const int f = idx_s[tl * K + j];
          first = !(f >= 0 && rank_of[f] == r);
        }
        if (first) key = r;
      }
    }
    row_s[i] = key;
    if (key >= 0) atomicAdd(reinterpret_cast<unsigned *>(&wh[key]), 1u);
  }
  __syncthreads();
  const int boff = p.do_expand ? 0 : E;
  for (int key = threadIdx.x; key < nkey; key += NT) {
    unsigned run = (unsigned)(seg_s[key] + bef_s[boff + key]);
    for (int w = 0; w < nrw; ++w) {
      const unsigned c = (unsigned)whist[(size_t)w * nkey + key];
      whist[(size_t)w * nkey + key] = run;
      run += c;
    }
  }
  __syncthreads();
  // Expanded layout: every slot owns its row, so pass 2 writes dst and the
  // row metadata directly; the rank layout resolves shared rows afterwards.
  int2 *meta = reinterpret_cast<int2 *>(p.meta);
  const unsigned lt = (1u << lane) - 1u;
  for (int s0 = beg; s0 < end; s0 += 32) {
    const int i = s0 + lane;
    const int key = i < end ? row_s[i] : -1;
    if (key >= 0) atomicOr(reinterpret_cast<unsigned *>(&wh[key]) + 1, 1u << lane);
    __syncwarp();
    const unsigned long long word = key >= 0 ? wh[key] : 0ull;
    const unsigned peers = (unsigned)(word >> 32);
    int row = -1;
    if (key >= 0) row = (int)((unsigned)word + __popc(peers & lt));
    __syncwarp();
    if (key >= 0 && lane == __ffs(peers) - 1)
      wh[key] = (unsigned long long)((unsigned)word + __popc(peers));
    __syncwarp();
    if (i < end) {
      if (p.do_expand) {
        bool keep = row >= 0 && row < p.row_limit;
        if (fcap > 0 && row >= 0 && row >= (key + 1) * fcap) keep = false;  // past capacity
        p.dst[base + i] = keep ? row : -1;
        if (keep) meta[row] = make_int2(t0 + i / K, i % K);
      } else {
        row_s[i] = row;
      }
    }
  }

  if (!p.do_expand) {
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += NT) {
      const int tl = i / K, k = i - tl * K;
      const int own = row_s[i];
      int row = own;
      const int e = idx_s[i];
      if (e >= 0 && own < 0) {
        // another (lower) slot of this token on the same rank owns the row
        const int r = rank_of[e];
        for (int j = 0; j < k; ++j) {
          const int f = idx_s[tl * K + j];
          if (f >= 0 && rank_of[f] == r) {
            row = row_s[tl * K + j];
            break;
          }
        }
      }
      if (row >= p.row_limit) row = -1;
      p.dst[base + i] = row;
      if (own >= 0 && own < p.row_limit) meta[own] = make_int2(t0 + tl, k);
    }
  }

  if (p.do_expand && fcap == 0 && b < p.num_blocks) {
    // alignment padding rows -> (-1, -1): one warp per expert, experts
    // b + (warp + NWARPS * i) * num_blocks over the ranking CTAs (the outputs
    // CTA has no segment starts)
    for (int e = b + warp * p.num_blocks; e < E; e += NWARPS * p.num_blocks) {
      const int64_t r0 = (int64_t)seg_s[e] + tot_s[e];
      const int64_t r1 = min((int64_t)seg_s[e + 1], p.row_limit);
      for (int64_t r = r0 + lane; r < r1; r += 32) meta[r] = make_int2(-1, -1);
    }
  }
}

}  // namespace

size_t layout_assign_smem(const LayoutParams &p) {
  const int nkey = p.do_expand ? p.E : p.R;
  return sizeof(int) * (2 * (size_t)p.chunk_tokens * p.K + 2 * (size_t)(p.E + p.R) + nkey + 1 +
                        p.E + 2 * (size_t)p.E + p.R + 1 + 1) +
         sizeof(unsigned long long) * (size_t)p.rank_warps * nkey;
}

int layout_rank_warps(int nkey) {
  // every warp ranks (a chunk has at most 8192 slots: 256 per warp); the
  // per-warp key histograms stay within ~48 KB of shared memory
  int w = NWARPS;
  while (w > 1 && (size_t)w * nkey * sizeof(unsigned long long) > 64 * 1024) w >>= 1;
  return w;
}

cudaError_t launch_layout(const LayoutParams &p, cudaStream_t s) {
  const size_t smem_count = sizeof(int) * (2 * (size_t)p.E + p.R + (size_t)p.chunk_tokens * p.K);
  const size_t smem_assign = layout_assign_smem(p);
  int dev = 0;
  cudaError_t err = launch_geometry(reinterpret_cast<const void *>(layout_count_kernel), NTC,
                                    smem_count, &dev, nullptr);
  if (err != cudaSuccess) return err;
  err = launch_geometry(reinterpret_cast<const void *>(layout_assign_kernel), NT, smem_assign,
                        &dev, nullptr);
  if (err != cudaSuccess) return err;
  layout_count_kernel<<<p.num_blocks, NTC, smem_count, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // assign may launch while count drains (programmatic dependent launch); it
  // waits on griddepcontrol before touching count's outputs
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(p.num_blocks + 1);  // + the outputs CTA
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = smem_assign;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, layout_assign_kernel, p);
}

}  // namespace ep
