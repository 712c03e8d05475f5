// Routing layout: counts, prefix sums, destination rows and source metadata.
//
// Follows the layout contract of "DeepEP V2 notes, ch. 7: how V2 dispatch
// builds expert inputs" (§7.2 layout metadata, §7.4 expanded layout) and the
// get_dispatch_layout outputs of the DeepEP README interface example.
//
// Tokens are cut into chunks of up to kLayoutChunkTokens tokens that never
// straddle a source rank.  A slot's row is
//     segment start of its key + its key's count in the chunks before
//                              + its stable rank among its chunk's slots
// (key = expert in the expanded layouts; in the rank layout, the rank, for
// the token's lowest slot on that rank).  Rows therefore ascend with
// (token, slot) inside every segment, and no atomic decides a position.  The
// last term depends on the chunk alone.  Two forms compute the same result:
//
// cluster form (rank layouts of at most kLayoutClusterChunks chunks): one
//   kernel, one CTA of 1024 threads per chunk plus one that owns no chunk,
//   the whole grid one thread-block cluster.  Each chunk CTA loads and
//   validates its chunk, counts experts and ranks (one thread per slot) in
//   shared memory, publishes the counts (cluster barrier arrival) and ranks
//   its slots; after the barrier it reads the other chunks' rank counts
//   through distributed shared memory, scans them into segment starts and
//   writes its rows.  The extra CTA sums every count over the chunks and
//   writes the global counts and prefix sums.
// two-kernel form (any size):
//   count  - one thread per token: validates and copies topk_idx, builds the
//            token's rank set (is_token_in_rank, first slot per rank) and
//            adds to the CTA's expert / rank histograms, stored block-major.
//   assign - every CTA sums the histogram columns it needs (global totals
//            and the totals of the chunks before it), scans them into segment
//            starts, then ranks its own slots.  One extra CTA, which owns no
//            chunk, writes the global counts and prefix sums (and, for the
//            host count wait, the mapped totals).
// Both rank slots the same way: warps walk contiguous runs of (token, slot)
// pairs in order, ranking equal keys with shared 64-bit words (a running
// count plus the mask of the lanes holding the key in the current step).
#include <algorithm>
#include <mutex>
#include <vector>

#include "ep_internal.cuh"
#include "ep_ptx.cuh"

namespace ep {
namespace {

constexpr int NT = kLayoutThreads;       // assign and cluster kernels: 1024 threads
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

// Exclusive scan of f(i), i < n, by the whole CTA of kThreads threads into
// out[0..n]; returns the total.  `warp_tot` is shared scratch of
// kThreads / 32 + 1 ints.
template <int kThreads, typename F>
__device__ int cta_exclusive_scan(int n, F f, int32_t *out, int *warp_tot) {
  constexpr int kWarps = kThreads / 32;
  if (n <= 32) {  // one warp's shuffle scan, one barrier
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int v = lane < n ? f(lane) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (lane < n) out[lane] = incl - v;
      if (lane == 31) out[n] = incl;
    }
    __syncthreads();
    return out[n];
  }
  if (n <= kThreads) {  // one value per thread: each warp adds up its own offset
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int v = (int)threadIdx.x < n ? f((int)threadIdx.x) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = lane; w < kWarps; w += 32) {
      const int t = warp_tot[w];
      total += t;
      before += w < warp ? t : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if ((int)threadIdx.x < n) out[threadIdx.x] = before + incl - v;
    if (threadIdx.x == 0) out[n] = total;
    __syncthreads();
    return total;
  }
  const int per = (n + kThreads - 1) / kThreads;
  const int beg = min((int)threadIdx.x * per, n);
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
    int w = lane < kWarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    if (lane < kWarps) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == kWarps - 1) warp_tot[kWarps] = wi;
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - local;
  for (int i = beg; i < end; ++i) {
    out[i] = run;
    run += f(i);
  }
  const int total = warp_tot[kWarps];
  if (threadIdx.x == 0) out[n] = total;
  __syncthreads();
  return total;
}

// Coalesced load of a chunk's ns topk_idx entries, eight loads in flight per
// thread.  Entries outside [-1, E) set EP_ERRBIT_BAD_TOPK_IDX and count as -1.
// Keeps an int32 copy in shared memory and in topk32; returns this thread's
// error bits.
template <int kThreads>
__device__ __forceinline__ unsigned load_chunk(const LayoutParams &p, int64_t base, int ns,
                                               int *idx_s) {
  unsigned err = 0;
  constexpr int kBatch = 8;
  for (int i0 = threadIdx.x; i0 < ns; i0 += kThreads * kBatch) {
    long long v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads;
      v[u] = -1;
      if (i < ns)
        v[u] = p.idx_is_int64 ? __ldg(static_cast<const long long *>(p.topk_idx) + base + i)
                              : __ldg(static_cast<const int *>(p.topk_idx) + base + i);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads;
      if (i >= ns) break;
      long long x = v[u];
      if (x < -1 || x >= p.E) {
        err |= EP_ERRBIT_BAD_TOPK_IDX;
        x = -1;
      }
      idx_s[i] = static_cast<int>(x);
      p.topk32[base + i] = static_cast<int>(x);
    }
  }
  return err;
}

// One thread per token (every thread of the CTA calls it; `active` is false
// past the chunk's end): adds the token's experts to hist_e and its rank set
// to hist_r, and writes its is_token_in_rank row.
__device__ __forceinline__ void token_pass(const LayoutParams &p, bool active, int64_t t,
                                           const int *trow, const int *rank_of, int *hist_e,
                                           int *hist_r) {
  const int K = p.K, R = p.R;
  const int lane = threadIdx.x & 31;
  uint64_t mask = 0;  // rank set (R <= 64)
  if (active) {
    for (int k = 0; k < K; ++k) {
      const int e = trow[k];
      if (e < 0) continue;
      atomicAdd(&hist_e[e], 1);
      const int r = rank_of[e];
      if (R <= 64) {
        mask |= 1ull << r;
      } else {  // wide rank sets: look back at this token's slots
        bool first = true;
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
    uint8_t *row = p.in_rank + t * R;
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
}

// Stable rank of the slots [beg, end) (one warp): key_s holds each slot's key
// (-1 for none); out(i, rank) receives, for every slot, the start held in
// its key's word plus its rank among the slots of the key from `beg` on (-1
// for no key).  The word of key k is wh[k * ws]; it holds that start in its
// low half, and its high half must be zero.  Every step takes 32 slots: each
// lane ORs its bit into its key's word, the word then names the lanes
// sharing the key (their order = slot order), and the lowest of them
// advances the key's running count.
template <typename Out>
__device__ __forceinline__ void rank_slots(int beg, int end, const int *key_s,
                                           unsigned long long *wh, int ws, Out out) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int s0 = beg; s0 < end; s0 += 32) {
    const int i = s0 + lane;
    const int key = i < end ? key_s[i] : -1;
    unsigned long long *w = wh + (size_t)(key >= 0 ? key : 0) * ws;
    if (key >= 0) atomicOr(reinterpret_cast<unsigned *>(w) + 1, 1u << lane);
    __syncwarp();
    const unsigned long long word = key >= 0 ? *w : 0ull;
    const unsigned peers = (unsigned)(word >> 32);
    int rank = -1;
    if (key >= 0) rank = (int)((unsigned)word + __popc(peers & lt));
    __syncwarp();
    if (key >= 0 && lane == __ffs(peers) - 1)
      *w = (unsigned long long)((unsigned)word + __popc(peers));
    __syncwarp();
    if (i < end) out(i, rank);
  }
}

// psum_rank_src[r][s], the tokens of source ranks < s that rank r receives,
// is the rank total of the chunks before source rank s's first chunk: that
// chunk's CTA holds it in bef_r.  Source ranks without tokens (and s = R) get
// the full total, written by the CTA with `empty_sources`.
template <int kThreads>
__device__ __forceinline__ void write_psum_rs(const LayoutParams &p, int b, const int *bef_r,
                                              const int *tot_r, bool empty_sources) {
  const int R = p.R, RR = R + 1;
  const int src_real = p.src_ranks;
  const int s = b / p.blocks_per_src;
  if (b < p.num_blocks && b == s * p.blocks_per_src && s < src_real)
    for (int r = threadIdx.x; r < R; r += kThreads) p.psum_rs[(int64_t)r * RR + s] = bef_r[r];
  if (empty_sources)
    for (int i = threadIdx.x; i < R * (RR - src_real); i += kThreads) {
      const int r = i / (RR - src_real), ss = src_real + (i - r * (RR - src_real));
      p.psum_rs[(int64_t)r * RR + ss] = tot_r[r];
    }
}

// Global outputs from the totals and the CTA-wide exclusive scan of
// [counts | aligned counts | rank counts] (prefix sums are read back by
// differences): counts, prefix sums, the dispatch counters, the control
// words and the host notification.  `err` is read in warp 0 only.
template <int kThreads>
__device__ __forceinline__ void write_outputs(const LayoutParams &p, const int *tot_s,
                                              const int32_t *scan_s, unsigned err) {
  static_assert(kThreads >= 96, "three warp roles");
  const int E = p.E, R = p.R, fcap = p.fixed_cap;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int a0 = scan_s[E], r0 = scan_s[2 * E];
  // Three warp roles side by side (the code of each runs once, so its
  // instruction fetches overlap those of the others): warp 0 the control
  // words (and the host's), warp 1 the rank outputs and the dispatch
  // counters, the other warps the expert outputs.
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
  } else if (warp == 1) {
    for (int r = lane; r <= R; r += 32) {
      if (r < R) p.cnt_r[r] = tot_s[E + r];
      p.psum_r[r] = scan_s[2 * E + r] - r0;
    }
    if (p.disp_sync != nullptr && lane < kDispSyncWords) p.disp_sync[lane] = 0;
  } else {
    for (int e = threadIdx.x - 64; e <= E; e += kThreads - 64) {
      const int pc = scan_s[e], pa = scan_s[E + e] - a0;
      if (e < E) {
        p.cnt_e[e] = tot_s[e];
        p.cnt_e_al[e] = scan_s[E + e + 1] - scan_s[E + e];  // aligned count
      }
      p.psum_e[e] = fcap > 0 ? pc : pa;  // fixed capacity: the prefix of the counts
      p.psum_pad[e] = pa - pc;
    }
  }
}

// Alignment padding rows of the aligned expanded layout -> (-1, -1): one warp
// per expert, experts b + (warp + kWarps * i) * nb.  seg(e) is the segment
// start of expert e (e <= E).
template <int kThreads, typename Seg>
__device__ __forceinline__ void write_padding(const LayoutParams &p, int b, int nb,
                                              const int *tot_s, Seg seg) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2 *meta = reinterpret_cast<int2 *>(p.meta);
  for (int e = b + warp * nb; e < p.E; e += kWarps * nb) {
    const int64_t r0 = (int64_t)seg(e) + tot_s[e];
    const int64_t r1 = min((int64_t)seg(e + 1), p.row_limit);
    for (int64_t r = r0 + lane; r < r1; r += 32) meta[r] = make_int2(-1, -1);
  }
}

// Column sums of per-chunk counts: for each key < nk, tot_s[key] = the sum
// over the nb chunks of column_of(key)(c) and bef_s[key] = the sum over the
// chunks before b.  g consecutive lanes share a key and split its chunks,
// eight loads in flight per lane.
template <int kThreads, typename ColumnOf>
__device__ __forceinline__ void column_sums(int nk, int nb, int b, ColumnOf column_of,
                                            int *tot_s, int *bef_s) {
  int g = 1;
  while (g < 32 && g * 2 * nk <= kThreads) g <<= 1;
  const int sub = threadIdx.x & (g - 1);
  const int per = kThreads / g;  // keys per pass
  for (int key0 = 0; key0 < nk; key0 += per) {
    const int key = key0 + (int)threadIdx.x / g;
    int tot = 0, bef = 0;
    if (key < nk) {
      const auto col = column_of(key);
      for (int bb = sub; bb < nb; bb += 8 * g) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = bb + u * g;
          v[u] = c < nb ? col(c) : 0;
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

// ---------------- cluster form (rank layout) ----------------

size_t cluster_head_ints(const LayoutParams &p) {
  return 6 * (size_t)p.E + 4 * (size_t)p.R + 2 + (size_t)p.chunk_tokens * p.K * 2;
}

// CTAs 0..nb-1 own the chunks; CTA nb, the last of the cluster, owns none and
// writes the global counts and prefix sums.
__global__ void __launch_bounds__(NT, 1) layout_cluster_kernel(LayoutParams p) {
  extern __shared__ __align__(16) int smem[];
  const int K = p.K, L = p.L, R = p.R, E = p.E, A = p.A;
  const int cap = p.chunk_tokens * K;
  const int nb = p.num_blocks;  // chunks; the grid is one cluster of nb + 1 CTAs
  const int nrw = p.rank_warps;
  // Read by the other CTAs of the cluster: this chunk's expert counts, rank
  // counts and error bits.
  int *pub = smem;                     // [E + R + 1]
  int *rank_of = pub + E + R + 1;      // [E] owning rank of each expert
  int *idx_s = rank_of + E;            // [cap]
  // [cap] per slot: the rank for the token's lowest slot on that rank (then
  // its rank among the chunk's such slots); -1 for an empty slot; -(j + 2)
  // for a slot whose row the token's lower slot j (chunk-relative) owns
  int *loc_s = idx_s + cap;
  int *tot_s = loc_s + cap;            // [E + R] totals over all chunks
  int *bef_s = tot_s + E + R;          // [E + R] totals of the chunks before this one
  int *scan_s = bef_s + E + R;         // [2E + R + 1]
  const int head = 6 * E + 4 * R + 2 + 2 * cap;
  // [R][nrw + 1] key words of the ranking ranges: key-major, so a warp
  // scans a key's ranges without bank conflicts; the odd row length spreads
  // the keys of one range (the atomics of the slot pass and the ranking)
  // over the banks
  const int kw = nrw + 1;
  unsigned long long *whist = reinterpret_cast<unsigned long long *>(smem + head + (head & 1));
  __shared__ int warp_tot[NWARPS + 1];

  const int b = blockIdx.x;
  const bool outputs_cta = b == nb;
  int t0 = p.T, nt = 0;
  if (!outputs_cta) nt = chunk_of(p, b, t0);
  const int ns = nt * K;
  const int64_t base = (int64_t)t0 * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // The chunk's topk_idx (ns <= 8 * NT) is requested first; the shared
  // memory and the is_token_in_rank rows are initialised while the loads are
  // in flight.
  long long v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = threadIdx.x + u * NT;
    v[u] = -1;
    if (i < ns)
      v[u] = p.idx_is_int64 ? __ldg(static_cast<const long long *>(p.topk_idx) + base + i)
                            : __ldg(static_cast<const int *>(p.topk_idx) + base + i);
  }
  for (int i = threadIdx.x; i < E + R + 1; i += NT) pub[i] = 0;
  for (int e = threadIdx.x; e < E; e += NT) rank_of[e] = e / L;
  for (int i = threadIdx.x; i < kw * R; i += NT) whist[i] = 0ull;
  uint8_t *in_rank = p.in_rank + (int64_t)t0 * R;
  if ((R & 3) == 0)
    for (int i = threadIdx.x; i < nt * R / 4; i += NT) reinterpret_cast<uint32_t *>(in_rank)[i] = 0;
  else
    for (int i = threadIdx.x; i < nt * R; i += NT) in_rank[i] = 0;
  // The next kernel (dispatch) may start its prologue; it waits for this
  // grid to complete before it reads anything written here.
  griddep_launch_dependents();
  unsigned err = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = threadIdx.x + u * NT;
    if (i < ns) {
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
  if (lane == 0 && err) atomicOr(reinterpret_cast<unsigned *>(&pub[E + R]), err);
  __syncthreads();

  // One thread per slot: the token's lowest slot on each rank (a look-back
  // over the token's slots) sets its is_token_in_rank byte and is the rank's
  // key, counted in its ranking range (warp w < nrw ranks the slots
  // [w * per, (w + 1) * per)); the expert and rank counts by shared atomics,
  // so the chunk's counts are published right after this pass.
  const int per = max(1, (ns + nrw - 1) / nrw);
  for (int i = threadIdx.x; i < ns; i += NT) {
    const int e = idx_s[i];
    int key = -1;
    if (e >= 0) {
      const int t = i / K, j0 = t * K;
      const int r = rank_of[e];
      int own = i;
      for (int j = j0; j < i; ++j) {
        const int f = idx_s[j];
        if (f >= 0 && rank_of[f] == r) {
          own = j;
          break;
        }
      }
      atomicAdd(&pub[e], 1);
      if (own == i) {
        in_rank[t * R + r] = 1;
        key = r;
        atomicAdd(&pub[E + r], 1);
        atomicAdd(reinterpret_cast<unsigned *>(&whist[(size_t)r * kw + i / per]), 1u);
      } else {
        key = -(own + 2);
      }
    }
    loc_s[i] = key;
  }
  __syncthreads();
  // This chunk's counts are published: the outputs CTA, which waits for
  // every chunk's, starts its sums and scan while the chunks rank their slots.
  cluster_arrive_release();
  // Each range's start per rank (warp per rank, lanes = ranges).
  for (int r = warp; r < R; r += NWARPS) {
    unsigned long long *wk = whist + (size_t)r * kw;
    const unsigned c = lane < nrw ? (unsigned)wk[lane] : 0u;
    unsigned incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nrw) wk[lane] = incl - c;
  }
  __syncthreads();

  // The in-order ranking overlaps the other chunks' arrival.
  if (warp < nrw)
    rank_slots(min(warp * per, ns), min((warp + 1) * per, ns), loc_s, whist + warp, kw,
               [&](int i, int rank) {
                 if (rank >= 0) loc_s[i] = rank;
               });
  __syncwarp();    // the cluster barriers are .aligned: whole warps
  cluster_wait();  // every chunk's counts are published

  if (outputs_cta) {
    // Column sums of every count over the chunks, one CTA-wide scan of
    // [counts | aligned counts | rank counts], the global outputs.
    column_sums<NT>(
        E + R, nb, b,
        [&](int key) {
          const uint32_t a = smem_u32(pub + key);
          return [a](int c) { return ld_cluster_s32(a, (uint32_t)c); };
        },
        tot_s, bef_s);
    unsigned err_all = 0;
    if (warp == 0)
      for (int c = lane; c < nb; c += 32)
        err_all |= (unsigned)ld_cluster_s32(smem_u32(pub + E + R), c);
    __syncwarp();
    cluster_arrive_relaxed();  // done reading the other CTAs' shared memory
    __syncthreads();
    cta_exclusive_scan<NT>(
        2 * E + R,
        [&](int i) {
          return i < E ? tot_s[i] : i < 2 * E ? (tot_s[i - E] + A - 1) / A * A : tot_s[i - E];
        },
        scan_s, warp_tot);
    write_outputs<NT>(p, tot_s, scan_s, err_all);
  } else {
    // The rank counts only: totals and the chunks before this one, then the
    // rank segment starts.
    column_sums<NT>(
        R, nb, b,
        [&](int key) {
          const uint32_t a = smem_u32(pub + E + key);
          return [a](int c) { return ld_cluster_s32(a, (uint32_t)c); };
        },
        tot_s + E, bef_s + E);
    __syncwarp();
    cluster_arrive_relaxed();  // done reading the other CTAs' shared memory
    __syncthreads();
    cta_exclusive_scan<NT>(R, [&](int r) { return tot_s[E + r]; }, scan_s, warp_tot);
    // the last chunk's CTA also writes the columns of source ranks without
    // tokens (from the rank totals), off the outputs CTA's path
    write_psum_rs<NT>(p, b, bef_s + E, tot_s + E, b == nb - 1);
    // Rows: segment start + the chunks before + the rank among the chunk's
    // slots; a slot whose row a lower slot of the token owns takes that row.
    int2 *meta = reinterpret_cast<int2 *>(p.meta);
    for (int i = threadIdx.x; i < ns; i += NT) {
      const int e = idx_s[i];
      const int loc = loc_s[i];
      int row = -1;
      if (loc >= 0) {
        const int r = rank_of[e];
        row = scan_s[r] + bef_s[E + r] + loc;
        if (row < p.row_limit) {
          const int t = i / K;
          meta[row] = make_int2(t0 + t, i - t * K);
        } else {
          row = -1;
        }
      } else if (loc <= -2) {
        const int r = rank_of[e];
        row = scan_s[r] + bef_s[E + r] + loc_s[-loc - 2];
        if (row >= p.row_limit) row = -1;
      }
      p.dst[base + i] = row;
    }
  }
  __syncwarp();
  cluster_wait();  // no CTA leaves while another may still read its counts
}

// ---------------- two-kernel form ----------------

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

  unsigned err = load_chunk<NTC>(p, base, ns, idx_s);
  err = __reduce_or_sync(0xffffffffu, err);
  __syncthreads();
  griddep_launch_dependents();  // the assign kernel's prologue may start now
  if (lane == 0 && err) atomicOr(&err_s, err);

  const int tl = threadIdx.x;
  token_pass(p, tl < nt, (int64_t)t0 + tl, idx_s + tl * K, rank_of, hist_e, hist_r);
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
  // offset.
  column_sums<NT>(
      E + R, p.num_blocks, b,
      [&](int key) {
        const int32_t *colp = key < E ? p.blk_e + key : p.blk_r + (key - E);
        const int stride = key < E ? E : R;
        return [colp, stride](int c) { return __ldcg(colp + (int64_t)c * stride); };
      },
      tot_s, bef_s);
  __syncthreads();
  write_psum_rs<NT>(p, b, bef_s + E, tot_s + E, b == p.num_blocks - 1);

  const int fcap = p.fixed_cap;
  if (b == p.num_blocks) {
    // The extra CTA that owns no chunk writes the global outputs (so no
    // ranking CTA waits for them).
    unsigned err = 0;
    if (warp == 0)  // issued before the scan, used after it
      for (int bb = lane; bb < p.num_blocks; bb += 32) err |= __ldcg(p.blk_err + bb);
    cta_exclusive_scan<NT>(
        2 * E + R,
        [&](int i) {
          return i < E ? tot_s[i] : i < 2 * E ? (tot_s[i - E] + A - 1) / A * A : tot_s[i - E];
        },
        scan_s, warp_tot);
    write_outputs<NT>(p, tot_s, scan_s, err);
    return;  // the outputs CTA ranks nothing
  }
  if (fcap > 0) {
    // Segment starts of the sort key: the fixed per-expert capacity, the
    // aligned expert counts, or the rank counts.
    for (int e = threadIdx.x; e <= E; e += NT) seg_s[e] = e * fcap;
    __syncthreads();
  } else if (p.do_expand) {
    cta_exclusive_scan<NT>(E, [&](int e) { return (tot_s[e] + A - 1) / A * A; }, seg_s, warp_tot);
  } else {
    cta_exclusive_scan<NT>(R, [&](int r) { return tot_s[E + r]; }, seg_s, warp_tot);
  }

  // Stable ranking: rank warp w owns the contiguous slot range [beg, end).
  // Pass 1 computes each slot's sort key -- the expert (expanded) or, for
  // the lowest slot of the token on each rank, the rank (rank layout) -- and
  // counts keys per warp (shared-memory atomics, order-free); after the
  // bases are known, pass 2 ranks the range in order.
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
  // With the bases folded into the words, the ranks are the rows.  Expanded
  // layout: every slot owns its row, so dst and the row metadata are written
  // at once; the rank layout resolves shared rows afterwards.
  int2 *meta = reinterpret_cast<int2 *>(p.meta);
  if (p.do_expand) {
    rank_slots(beg, end, row_s, wh, 1, [&](int i, int row) {
      bool keep = row >= 0 && row < p.row_limit;
      if (fcap > 0 && keep && row >= (idx_s[i] + 1) * fcap) keep = false;  // past capacity
      p.dst[base + i] = keep ? row : -1;
      if (keep) meta[row] = make_int2(t0 + i / K, i % K);
    });
  } else {
    rank_slots(beg, end, row_s, wh, 1, [&](int i, int row) { row_s[i] = row; });
    __syncthreads();
  }

  for (int i = threadIdx.x; i < ns && !p.do_expand; i += NT) {
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

  if (p.do_expand && fcap == 0)
    write_padding<NT>(p, b, p.num_blocks, tot_s, [&](int e) { return seg_s[e]; });
}

size_t cluster_smem(const LayoutParams &p) {
  const size_t head = cluster_head_ints(p);
  return sizeof(int) * (head + (head & 1)) +
         sizeof(unsigned long long) * (size_t)(p.rank_warps + 1) * p.R;
}

// Whether a cluster of `nb` CTAs of the cluster kernel at `smem` bytes can be
// launched on the current device (looked up once per device and shape).
cudaError_t cluster_launchable(int nb, size_t smem, bool *ok) {
  struct Entry {
    int device, nb;
    size_t smem;
    bool ok;
  };
  static std::mutex mu;
  static std::vector<Entry> shapes;
  int dev = 0;
  cudaError_t err =
      launch_geometry(reinterpret_cast<const void *>(layout_cluster_kernel), NT, smem, &dev,
                      nullptr);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> g(mu);
  for (const Entry &e : shapes)
    if (e.device == dev && e.nb == nb && e.smem == smem) {
      *ok = e.ok;
      return cudaSuccess;
    }
  if (nb > 8) {
    err = cudaFuncSetAttribute(layout_cluster_kernel,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(nb);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nb;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, layout_cluster_kernel, &lc);
  if (err != cudaSuccess) {
    cudaGetLastError();  // not launchable as a cluster: use the two-kernel form
    clusters = 0;
  }
  *ok = clusters > 0;
  shapes.push_back({dev, nb, smem, *ok});
  return cudaSuccess;
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

cudaError_t launch_layout(const LayoutParams &p, cudaStream_t s, int *kernels) {
  *kernels = 0;
  const size_t smem_cl = cluster_smem(p);
  // The cluster form measured faster than the two kernels for the rank
  // layout only (decode: 14.3 against 15.0 us per layout); the expanded
  // layouts keep two kernels.
  if (!p.do_expand && p.num_blocks <= kLayoutClusterChunks && smem_cl <= kLayoutClusterSmem) {
    bool ok = false;
    cudaError_t err = cluster_launchable(p.num_blocks + 1, smem_cl, &ok);
    if (err != cudaSuccess) return err;
    if (ok) {
      cudaLaunchConfig_t lc{};
      lc.gridDim = dim3(p.num_blocks + 1);  // + the outputs CTA
      lc.blockDim = dim3(NT);
      lc.dynamicSmemBytes = smem_cl;
      lc.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = p.num_blocks + 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      lc.attrs = attr;
      lc.numAttrs = 1;
      *kernels = 1;
      return cudaLaunchKernelEx(&lc, layout_cluster_kernel, p);
    }
  }
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
  *kernels = 2;
  return cudaLaunchKernelEx(&lc, layout_assign_kernel, p);
}

}  // namespace ep
