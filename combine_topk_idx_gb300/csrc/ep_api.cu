// Host side of libep.so: argument checks, sizing, handle ownership, launches.
//
// The contract (who allocates what, exact vs upper-bound sizes, handle
// contents) follows "DeepEP V2 notes, ch. 7: how V2 dispatch builds expert
// inputs" §7.1, §7.2 and §7.5, and "ch. 8: combine, handle and async
// overlap" §8.1 / §8.2 (everything is ordered on the caller's stream).
#include <chrono>
#include <mutex>
#include <thread>
#include <vector>

#include "ep_internal.cuh"

struct ep_handle {
  ep_config cfg;
  int device;
  cudaStream_t stream;
  void *dmem;
  ep::LayoutParams lp;
  int64_t rows_alloc;
  int64_t sf_hidden_stride, sf_token_stride, sf_numel, sf_expert_stride;
  float *tok_scale;
};

namespace ep {

int device_sm_count(int device) {
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> g(mu);
  if (device < 0) return 1;
  if ((int)cache.size() <= device) cache.resize(device + 1, 0);
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
      n = 1;
    cache[device] = n;
  }
  return cache[device];
}

cudaError_t launch_geometry(const void *func, int threads, size_t smem, int *device,
                            int *per_sm) {
  struct Entry {
    const void *func;
    int device, threads;
    size_t smem;
    int per_sm;
  };
  struct OptIn {
    const void *func;
    int device;
    size_t smem;  // largest dynamic shared memory opted in so far
  };
  static std::mutex mu;
  static std::vector<Entry> shapes;
  static std::vector<OptIn> optins;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  *device = dev;
  std::lock_guard<std::mutex> g(mu);
  if (per_sm != nullptr)
    for (const Entry &e : shapes)
      if (e.func == func && e.device == dev && e.threads == threads && e.smem == smem) {
        *per_sm = e.per_sm;
        return cudaSuccess;
      }
  if (smem > kDynSmemOptIn) {
    OptIn *o = nullptr;
    for (OptIn &x : optins)
      if (x.func == func && x.device == dev) o = &x;
    if (o == nullptr || o->smem < smem) {
      err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      if (o == nullptr)
        optins.push_back({func, dev, smem});
      else
        o->smem = smem;
    }
  }
  if (per_sm == nullptr) return cudaSuccess;  // the opt-in only
  int n = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
  if (err != cudaSuccess) return err;
  shapes.push_back({func, dev, threads, smem, n});
  *per_sm = n;
  return cudaSuccess;
}

namespace {

// Host waits poll without yielding the CPU for this long, then yield between
// polls.
constexpr int kTightPollMs = 2;

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Bounds {
  int64_t per_rank, global, rows;
};

Bounds upper_bound(const ep_config &c) {
  const int64_t T = c.num_tokens, K = c.num_topk, E = c.num_experts, R = c.num_ranks;
  const int64_t L = E / R, M = c.num_max_tokens_per_rank, A = c.expert_alignment;
  Bounds b;
  if (c.fixed_capacity) {  // every expert owns M * R rows, whatever the counts
    b.per_rank = L * M * R;
    b.global = E * M * R;
    b.rows = b.global;
    return b;
  }
  if (c.do_expand) {
    b.per_rank = align_up(R * M * std::min(K, L) + (A - 1) * L, A);
    b.global = align_up(T * K + E * (A - 1), A);
  } else {
    b.per_rank = M * R;
    b.global = T * std::min(K, R);
  }
  b.rows = std::min(R * b.per_rank, b.global);
  return b;
}

// Polls the three tagged words of `slot` until each carries `seq` (or the
// deadline passes); returns their values in words[0..2].  The first
// kTightPollMs are polled without yielding the CPU: a caller whose call was
// enqueued behind other GPU work often waits that long, and a yield between
// polls adds to the reaction once the words land (prefill step -1.7 us).
ep_status wait_host_words(const HostSync *slot, int32_t seq, int32_t timeout_ms,
                          uint64_t words[3]) {
  const uint64_t tag = (uint64_t)(uint32_t)seq;
  const volatile uint64_t *src[3] = {&slot->num_recv, &slot->num_expanded, &slot->error};
  const auto start = std::chrono::steady_clock::now();
  const auto deadline = start + std::chrono::milliseconds(timeout_ms);
  bool long_wait = false;
  int got = 0;
  for (uint64_t spin = 0;; ++spin) {
    while (got < 3) {
      const uint64_t v =
          __atomic_load_n(const_cast<const uint64_t *>(src[got]), __ATOMIC_ACQUIRE);
      if ((v >> 32) != tag) break;
      words[got++] = v;
    }
    if (got == 3) return EP_OK;
    if ((spin & 255) == 0) {
      const auto now = std::chrono::steady_clock::now();
      if (now >= deadline) return EP_ERR_TIMEOUT;
      long_wait = now - start > std::chrono::milliseconds(kTightPollMs);
    }
    if (long_wait) std::this_thread::yield();
  }
}

// Pool of pinned, device-mapped host words for the count wait.  Each slot
// keeps the device address of its mapping, looked up once per block of slots.
struct SyncPool {
  struct Slot {
    HostSync *host;
    HostSync *dev;
  };
  std::mutex mu;
  std::vector<Slot> free_list;
  int32_t seq = 0;
  bool acquire(int32_t *seq_out, Slot *out) {
    std::lock_guard<std::mutex> g(mu);
    *seq_out = ++seq;
    if (seq > 0x3fffffff) seq = 0;
    if (free_list.empty()) {
      const int n = 64;
      void *mem = nullptr;
      if (cudaHostAlloc(&mem, n * sizeof(HostSync), cudaHostAllocMapped | cudaHostAllocPortable) !=
          cudaSuccess)
        return false;
      void *dmem = nullptr;
      if (cudaHostGetDevicePointer(&dmem, mem, 0) != cudaSuccess) {
        cudaFreeHost(mem);
        return false;
      }
      HostSync *s = static_cast<HostSync *>(mem);
      HostSync *d = static_cast<HostSync *>(dmem);
      for (int i = 0; i < n; ++i) free_list.push_back({s + i, d + i});
    }
    *out = free_list.back();
    free_list.pop_back();
    return true;
  }
  void release(const Slot &h) {
    std::lock_guard<std::mutex> g(mu);
    free_list.push_back(h);
  }
};

SyncPool &sync_pool() {
  static SyncPool *p = new SyncPool();  // never destroyed: kernels may still hold slots at exit
  return *p;
}

// A memory pool per device for handle metadata: freed blocks are kept for
// reuse (release threshold = max), so steady-state ep_layout calls do not map
// new device memory.  Lives until process exit.
cudaError_t handle_pool(int device, cudaMemPool_t *out) {
  static std::mutex mu;
  static std::vector<cudaMemPool_t> pools;
  std::lock_guard<std::mutex> g(mu);
  if ((int)pools.size() <= device) pools.resize(device + 1, nullptr);
  if (pools[device] == nullptr) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t threshold = ~0ull;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &threshold);
    if (e != cudaSuccess) return e;
    pools[device] = pool;
  }
  *out = pools[device];
  return cudaSuccess;
}

ep_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return EP_OK;
  if (e == cudaErrorMemoryAllocation) return EP_ERR_OOM;
  return EP_ERR_CUDA;
}

}  // namespace
}  // namespace ep

using ep::align_up;
using ep::aligned;

namespace ep {
namespace {

ep_status check_device(const ep_handle *h) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
  return dev == h->device ? EP_OK : EP_ERR_INVALID_ARG;
}

DispatchParams dispatch_params(const ep_handle *h, const void *x, const float *topk_weights,
                               void *recv_x, float *recv_sf, float *recv_topk_weights,
                               int32_t *recv_topk_idx) {
  const ep_config &c = h->cfg;
  DispatchParams p{};
  p.x = static_cast<const uint16_t *>(x);
  p.topk_w = topk_weights;
  p.topk32 = h->lp.topk32;
  p.dst = h->lp.dst;
  p.psum_e = h->lp.psum_e;
  p.cnt_e = h->lp.cnt_e;
  p.psum_pad = h->lp.psum_pad;
  p.T = c.num_tokens;
  p.K = c.num_topk;
  p.E = c.num_experts;
  p.L = c.num_experts / c.num_ranks;
  p.H = c.hidden;
  p.do_expand = c.do_expand;
  p.zero_padding = c.do_expand && c.do_zero_padding;
  p.max_pad_items = c.do_expand ? ((int64_t)c.num_experts * (c.expert_alignment - 1) + 7) / 8 : 0;
  p.rows_alloc = h->rows_alloc;
  p.sf_hidden_stride = h->sf_hidden_stride;
  p.sf_token_stride = h->sf_token_stride;
  p.recv_x = recv_x;
  p.recv_sf = recv_sf;
  p.recv_w = recv_topk_weights;
  p.recv_idx = recv_topk_idx;
  p.err = reinterpret_cast<unsigned *>(h->lp.ctrl + kCtrlError);
  p.tok_scale = h->tok_scale;
  p.meta = h->lp.meta;
  p.num_rows = h->lp.ctrl + (c.do_expand ? kCtrlNumExpanded : kCtrlNumRecv);
  p.sf_src = h->tok_scale;
  p.sf_src_ts = c.hidden / 128;
  p.sf_src_hs = 1;
  p.fixed_cap = h->lp.fixed_cap;
  p.sf_expert_stride = h->sf_expert_stride;
  p.sf_sync = h->lp.disp_sync;
  p.sched = h->lp.disp_sync + 2;
  return p;
}

CombineParams combine_params(const ep_handle *h, const void *y, const float *topk_weights,
                             const void *bias_0, const void *bias_1, const void *expert_bias,
                             void *out) {
  const ep_config &c = h->cfg;
  CombineParams p{};
  p.y = static_cast<const uint16_t *>(y);
  p.topk_w = topk_weights;
  p.topk32 = h->lp.topk32;
  p.dst = h->lp.dst;
  p.bias0 = static_cast<const uint16_t *>(bias_0);
  p.bias1 = static_cast<const uint16_t *>(bias_1);
  p.ebias = static_cast<const uint16_t *>(expert_bias);
  p.out = static_cast<uint16_t *>(out);
  p.err = reinterpret_cast<unsigned *>(h->lp.ctrl + kCtrlError);
  p.T = c.num_tokens;
  p.K = c.num_topk;
  p.H = c.hidden;
  p.rows_alloc = h->rows_alloc;
  return p;
}

}  // namespace
}  // namespace ep

extern "C" {

const char *ep_status_string(ep_status s) {
  switch (s) {
    case EP_OK: return "ok";
    case EP_ERR_INVALID_ARG: return "invalid argument";
    case EP_ERR_UNSUPPORTED: return "unsupported configuration";
    case EP_ERR_BAD_TOPK_IDX: return "topk_idx value outside [-1, num_experts)";
    case EP_ERR_CUDA: return "CUDA runtime error";
    case EP_ERR_OOM: return "out of memory";
    case EP_ERR_TIMEOUT: return "timed out waiting for the receive counts";
    case EP_ERR_OVERFLOW: return "upper-bound allocation exceeded";
  }
  return "unknown status";
}

int32_t ep_abi_version(void) { return EP_ABI_VERSION; }

ep_status ep_validate_config(const ep_config *c) {
  if (c == nullptr) return EP_ERR_INVALID_ARG;
  if (c->num_tokens < 0 || c->num_topk < 1 || c->num_experts < 1 || c->num_ranks < 1 ||
      c->hidden < 1 || c->num_max_tokens_per_rank < 1 || c->expert_alignment < 1 ||
      c->num_sms < 0 || c->cpu_sync_timeout_ms < 0)
    return EP_ERR_INVALID_ARG;
  if (c->num_experts % c->num_ranks != 0) return EP_ERR_INVALID_ARG;
  if (c->hidden % 8 != 0) return EP_ERR_INVALID_ARG;
  if (c->use_fp8 && c->hidden % 128 != 0) return EP_ERR_INVALID_ARG;
  if ((int64_t)c->num_tokens > (int64_t)c->num_max_tokens_per_rank * c->num_ranks)
    return EP_ERR_INVALID_ARG;
  if (c->topk_idx_is_int64 != 0 && c->topk_idx_is_int64 != 1) return EP_ERR_INVALID_ARG;
  if (c->do_expand > 1 || c->do_zero_padding > 1 || c->do_cpu_sync > 1 || c->use_fp8 > 1 ||
      c->use_tma_aligned_col_major_sf > 1 || c->fixed_capacity > 1)
    return EP_ERR_INVALID_ARG;
  if (c->reserved0[0] | c->reserved0[1]) return EP_ERR_INVALID_ARG;
  // the fixed-capacity layout is expanded, unaligned and has no padding
  if (c->fixed_capacity &&
      (!c->do_expand || c->expert_alignment != 1 || c->do_zero_padding))
    return EP_ERR_INVALID_ARG;
  if (c->num_topk > EP_MAX_TOPK || c->num_experts > EP_MAX_EXPERTS || c->hidden > EP_MAX_HIDDEN)
    return EP_ERR_UNSUPPORTED;
  const ep::Bounds b = ep::upper_bound(*c);
  const int64_t lim = 0x7fffffffLL;
  if ((int64_t)c->num_tokens * c->num_topk > lim || b.global > lim ||
      (int64_t)c->num_tokens * c->num_ranks > (int64_t)1 << 40)
    return EP_ERR_UNSUPPORTED;
  return EP_OK;
}

ep_status ep_upper_bound_rows(const ep_config *cfg, int64_t *rows) {
  if (rows == nullptr) return EP_ERR_INVALID_ARG;
  const ep_status st = ep_validate_config(cfg);
  if (st != EP_OK) return st;
  *rows = ep::upper_bound(*cfg).rows;
  return EP_OK;
}

ep_status ep_host_wait_flag(const volatile int32_t *flag, int32_t expected, int32_t timeout_ms) {
  if (flag == nullptr || timeout_ms < 0) return EP_ERR_INVALID_ARG;
  const auto start = std::chrono::steady_clock::now();
  const auto deadline = start + std::chrono::milliseconds(timeout_ms);
  bool long_wait = false;
  for (uint64_t spin = 0;; ++spin) {
    if (__atomic_load_n(const_cast<const int32_t *>(flag), __ATOMIC_ACQUIRE) == expected)
      return EP_OK;
    if ((spin & 255) == 0) {
      const auto now = std::chrono::steady_clock::now();
      if (now >= deadline) return EP_ERR_TIMEOUT;
      long_wait = now - start > std::chrono::milliseconds(ep::kTightPollMs);
    }
    if (long_wait) std::this_thread::yield();
  }
}

namespace ep {
namespace {

// Scale-factor strides and size of a handle with `rows_alloc` receive rows.
void plan_sf(const ep_config &c, int64_t rows_alloc, int64_t fixed_cap, int64_t *token_stride,
             int64_t *hidden_stride, int64_t *numel, int64_t *expert_stride) {
  const int64_t nb = c.hidden / kFp8Block;
  *expert_stride = 0;
  if (c.use_fp8 && c.fixed_capacity) {
    if (c.use_tma_aligned_col_major_sf) {  // one column-major slab per expert
      *token_stride = 1;
      *hidden_stride = align_up(fixed_cap, 4);
      *expert_stride = nb * *hidden_stride;
    } else {
      *token_stride = nb;
      *hidden_stride = 1;
      *expert_stride = nb * fixed_cap;
    }
    *numel = (int64_t)c.num_experts * *expert_stride;
  } else if (c.use_fp8) {
    if (c.use_tma_aligned_col_major_sf) {
      *token_stride = 1;
      *hidden_stride = align_up(rows_alloc, 4);
      *numel = nb * *hidden_stride;
    } else {
      *token_stride = nb;
      *hidden_stride = 1;
      *numel = nb * rows_alloc;
    }
  } else {
    *token_stride = *hidden_stride = *numel = 0;
  }
}

// Everything of a layout up to its launch: checks, the layout parameters and
// the handle's device block (stream-ordered on s).
struct LayoutSetup {
  ep_config c;
  cudaStream_t s;
  bool capturing;
  int dev;
  Bounds b;
  LayoutParams lp;
  void *dmem;
  float *tok_scale;
};

ep_status layout_setup(const ep_config *cfg, const void *topk_idx, ep_stream_t stream,
                       LayoutSetup *L) {
  ep_status st = ep_validate_config(cfg);
  if (st != EP_OK) return st;
  const ep_config c = *cfg;
  L->c = c;
  const int T = c.num_tokens, K = c.num_topk, E = c.num_experts, R = c.num_ranks;
  if (T > 0 && (topk_idx == nullptr || !aligned(topk_idx, c.topk_idx_is_int64 ? 8 : 4)))
    return EP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  L->s = s;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return EP_ERR_CUDA;
  L->capturing = cs != cudaStreamCaptureStatusNone;
  if (c.do_cpu_sync && L->capturing) return EP_ERR_INVALID_ARG;
  if (cudaGetDevice(&L->dev) != cudaSuccess) return EP_ERR_CUDA;

  const Bounds b = upper_bound(c);
  L->b = b;
  LayoutParams lp{};
  lp.topk_idx = topk_idx;
  lp.idx_is_int64 = c.topk_idx_is_int64;
  lp.T = T; lp.K = K; lp.E = E; lp.R = R; lp.L = E / R;
  lp.M = c.num_max_tokens_per_rank;
  lp.A = c.expert_alignment;
  lp.do_expand = c.do_expand;
  lp.fixed_cap = c.fixed_capacity ? c.num_max_tokens_per_rank * c.num_ranks : 0;
  // exact mode: rows never exceed the global bound; upper-bound mode: rows
  // past the allocation are dropped and flagged
  lp.row_limit = c.do_cpu_sync ? b.global : b.rows;
  // Chunks of up to 256 tokens that never straddle a source rank.
  lp.chunk_tokens = kLayoutChunkTokens;
  const int TB = lp.chunk_tokens;
  const int64_t src_ranks = ((int64_t)T + lp.M - 1) / lp.M;
  const int64_t max_tok = std::min<int64_t>(lp.M, T);
  lp.blocks_per_src = (int)std::max<int64_t>(1, (max_tok + TB - 1) / TB);
  const int64_t nblocks = std::max<int64_t>(1, src_ranks * lp.blocks_per_src);
  if (nblocks > 0x7fffffff) return EP_ERR_UNSUPPORTED;
  lp.num_blocks = (int)nblocks;
  lp.src_ranks = (int)src_ranks;
  lp.rank_warps = layout_rank_warps(c.do_expand ? E : R);
  if (layout_assign_smem(lp) > 220 * 1024) return EP_ERR_UNSUPPORTED;

  // One device block, carved into 256-byte aligned arrays.
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t o_ctrl = take(sizeof(int32_t) * kCtrlWords);
  const size_t o_sync = take(sizeof(int32_t) * kDispSyncWords);
  const size_t o_topk = take(sizeof(int32_t) * (size_t)T * K);
  const size_t o_dst = take(sizeof(int32_t) * (size_t)T * K);
  const size_t o_meta = take(sizeof(int32_t) * 2 * (size_t)lp.row_limit);
  const size_t o_inr = take((size_t)T * R);
  const size_t o_cnte = take(sizeof(int32_t) * E);
  const size_t o_cntea = take(sizeof(int32_t) * E);
  const size_t o_pse = take(sizeof(int32_t) * (E + 1));
  const size_t o_psp = take(sizeof(int32_t) * (E + 1));
  const size_t o_cntr = take(sizeof(int32_t) * R);
  const size_t o_psr = take(sizeof(int32_t) * (R + 1));
  const size_t o_psrs = take(sizeof(int32_t) * (size_t)R * (R + 1));
  const size_t o_blke = take(sizeof(int32_t) * (size_t)E * lp.num_blocks);
  const size_t o_blkr = take(sizeof(int32_t) * (size_t)R * lp.num_blocks);
  const size_t o_blkerr = take(sizeof(uint32_t) * (size_t)lp.num_blocks);
  const size_t o_toks = take(c.use_fp8 ? sizeof(float) * (size_t)T * (c.hidden / kFp8Block) : 0);
  void *dmem = nullptr;
  cudaError_t ce;
  if (L->capturing) {
    // inside a stream capture the allocation becomes a graph memory node
    ce = cudaMallocAsync(&dmem, off, s);
  } else {
    cudaMemPool_t pool = nullptr;
    ce = handle_pool(L->dev, &pool);
    if (ce == cudaSuccess) ce = cudaMallocFromPoolAsync(&dmem, off, pool, s);
  }
  if (ce != cudaSuccess) return cuda_status(ce);
  uint8_t *base = static_cast<uint8_t *>(dmem);
  lp.ctrl = reinterpret_cast<int32_t *>(base + o_ctrl);
  lp.disp_sync = reinterpret_cast<int32_t *>(base + o_sync);
  lp.topk32 = reinterpret_cast<int32_t *>(base + o_topk);
  lp.dst = reinterpret_cast<int32_t *>(base + o_dst);
  lp.meta = reinterpret_cast<int32_t *>(base + o_meta);
  lp.in_rank = base + o_inr;
  lp.cnt_e = reinterpret_cast<int32_t *>(base + o_cnte);
  lp.cnt_e_al = reinterpret_cast<int32_t *>(base + o_cntea);
  lp.psum_e = reinterpret_cast<int32_t *>(base + o_pse);
  lp.psum_pad = reinterpret_cast<int32_t *>(base + o_psp);
  lp.cnt_r = reinterpret_cast<int32_t *>(base + o_cntr);
  lp.psum_r = reinterpret_cast<int32_t *>(base + o_psr);
  lp.psum_rs = reinterpret_cast<int32_t *>(base + o_psrs);
  lp.blk_e = reinterpret_cast<int32_t *>(base + o_blke);
  lp.blk_r = reinterpret_cast<int32_t *>(base + o_blkr);
  lp.blk_err = reinterpret_cast<uint32_t *>(base + o_blkerr);
  L->tok_scale = c.use_fp8 ? reinterpret_cast<float *>(base + o_toks) : nullptr;
  L->lp = lp;
  L->dmem = dmem;
  return EP_OK;
}

// The handle of a launched layout with `rows_alloc` receive rows.
ep_handle *make_handle(const LayoutSetup &L, int64_t rows_alloc) {
  ep_handle *h = new ep_handle();
  h->cfg = L.c;
  h->device = L.dev;
  h->stream = L.s;
  h->dmem = L.dmem;
  h->lp = L.lp;
  h->lp.host = nullptr;
  h->lp.topk_idx = nullptr;
  h->tok_scale = L.tok_scale;
  h->rows_alloc = rows_alloc;
  plan_sf(L.c, rows_alloc, L.lp.fixed_cap, &h->sf_token_stride, &h->sf_hidden_stride,
          &h->sf_numel, &h->sf_expert_stride);
  return h;
}

void fill_info(const ep_handle *h, int64_t num_recv, int64_t num_exp, int layout_kernels,
               ep_layout_info *info) {
  const LayoutParams &lp = h->lp;
  info->num_recv_tokens = num_recv;
  info->num_expanded_tokens = num_exp;
  info->rows_alloc = h->rows_alloc;
  info->sf_numel = h->sf_numel;
  info->sf_token_stride = h->sf_token_stride;
  info->sf_hidden_stride = h->sf_hidden_stride;
  info->topk_idx = lp.topk32;
  info->cnt_expert = lp.cnt_e;
  info->cnt_expert_aligned = lp.cnt_e_al;
  info->psum_expert = lp.psum_e;
  info->cnt_rank = lp.cnt_r;
  info->psum_rank = lp.psum_r;
  info->psum_rank_src = lp.psum_rs;
  info->dst_buffer_slot_idx = lp.dst;
  info->recv_src_metadata = lp.meta;
  info->is_token_in_rank = lp.in_rank;
  info->totals = lp.ctrl + kCtrlNumRecv;
  info->error_word = reinterpret_cast<const uint32_t *>(lp.ctrl + kCtrlError);
  info->meta_rows = lp.row_limit;
  info->expert_capacity = lp.fixed_cap;
  info->sf_expert_stride = h->sf_expert_stride;
  info->layout_kernels = layout_kernels;
  info->reserved1 = 0;
}

}  // namespace
}  // namespace ep

ep_status ep_layout(const ep_config *cfg, const void *topk_idx, ep_stream_t stream,
                    ep_handle **out_handle, ep_layout_info *info) {
  if (out_handle == nullptr || info == nullptr) return EP_ERR_INVALID_ARG;
  *out_handle = nullptr;
  ep::LayoutSetup L;
  ep_status st = ep::layout_setup(cfg, topk_idx, stream, &L);
  if (st != EP_OK) return st;
  const ep_config &c = L.c;
  ep::LayoutParams &lp = L.lp;
  auto fail = [&](ep_status code) {
    cudaFreeAsync(L.dmem, L.s);
    return code;
  };

  ep::SyncPool::Slot slot{nullptr, nullptr};
  if (c.do_cpu_sync) {
    int32_t seq = 0;
    if (!ep::sync_pool().acquire(&seq, &slot)) return fail(EP_ERR_OOM);
    slot.host->num_recv = slot.host->num_expanded = slot.host->error = 0;
    lp.host = slot.dev;
    lp.seq = seq;
  }
  int layout_kernels = 0;
  const cudaError_t ce = ep::launch_layout(lp, L.s, &layout_kernels);
  if (ce != cudaSuccess) {
    // the kernel may not have run: the slot is not safe to hand out again
    return fail(ep::cuda_status(ce));
  }

  st = EP_OK;
  int64_t num_recv = -1, num_exp = -1;
  int64_t rows_alloc = L.b.rows;
  if (c.do_cpu_sync) {
    const int32_t timeout = c.cpu_sync_timeout_ms > 0 ? c.cpu_sync_timeout_ms : 10000;
    uint64_t words[3];
    const ep_status w = ep::wait_host_words(slot.host, lp.seq, timeout, words);
    if (w != EP_OK) {
      // the slot may still be written later: leave it out of the pool
      return fail(w);
    }
    num_recv = (uint32_t)words[0];
    num_exp = (uint32_t)words[1];
    const uint32_t err = (uint32_t)words[2];
    ep::sync_pool().release(slot);
    rows_alloc = c.fixed_capacity ? L.b.rows : c.do_expand ? num_exp : num_recv;
    if (err & EP_ERRBIT_BAD_TOPK_IDX) st = EP_ERR_BAD_TOPK_IDX;
  }
  ep_handle *h = ep::make_handle(L, rows_alloc);
  ep::fill_info(h, num_recv, num_exp, layout_kernels, info);
  *out_handle = h;
  return st;
}

ep_status ep_plan_layout(const ep_config *cfg, ep_layout_info *info) {
  if (info == nullptr) return EP_ERR_INVALID_ARG;
  const ep_status st = ep_validate_config(cfg);
  if (st != EP_OK) return st;
  if (cfg->do_cpu_sync) return EP_ERR_INVALID_ARG;  // sizes depend on the routing
  const ep::Bounds b = ep::upper_bound(*cfg);
  const int64_t fixed_cap =
      cfg->fixed_capacity ? (int64_t)cfg->num_max_tokens_per_rank * cfg->num_ranks : 0;
  *info = ep_layout_info{};
  info->num_recv_tokens = info->num_expanded_tokens = -1;
  info->rows_alloc = b.rows;
  ep::plan_sf(*cfg, b.rows, fixed_cap, &info->sf_token_stride, &info->sf_hidden_stride,
              &info->sf_numel, &info->sf_expert_stride);
  info->meta_rows = b.rows;
  info->expert_capacity = fixed_cap;
  return EP_OK;
}

namespace ep {
namespace {

// Pointer checks of a quantising / BF16 dispatch into `rows_alloc` rows.
ep_status check_dispatch_args(const ep_config &c, int64_t rows_alloc, const void *x,
                              const float *topk_weights, const void *recv_x,
                              const float *recv_sf, const float *recv_topk_weights,
                              const int32_t *recv_topk_idx) {
  const int T = c.num_tokens;
  if (T > 0 && (x == nullptr || !aligned(x, 16))) return EP_ERR_INVALID_ARG;
  if (rows_alloc > 0 && (recv_x == nullptr || !aligned(recv_x, 16))) return EP_ERR_INVALID_ARG;
  if (c.use_fp8) {
    if (rows_alloc > 0 && (recv_sf == nullptr || !aligned(recv_sf, 4))) return EP_ERR_INVALID_ARG;
  } else if (recv_sf != nullptr) {
    return EP_ERR_INVALID_ARG;
  }
  if (recv_topk_weights != nullptr &&
      ((T > 0 && topk_weights == nullptr) || !aligned(recv_topk_weights, 4)))
    return EP_ERR_INVALID_ARG;
  if (topk_weights != nullptr && !aligned(topk_weights, 4)) return EP_ERR_INVALID_ARG;
  if (recv_topk_idx != nullptr && (c.do_expand || !aligned(recv_topk_idx, 4)))
    return EP_ERR_INVALID_ARG;
  return EP_OK;
}

}  // namespace
}  // namespace ep

ep_status ep_dispatch(ep_handle *h, const void *x, const float *topk_weights, void *recv_x,
                      float *recv_sf, float *recv_topk_weights, int32_t *recv_topk_idx,
                      ep_stream_t stream) {
  if (h == nullptr) return EP_ERR_INVALID_ARG;
  const ep_config &c = h->cfg;
  if (const ep_status st = ep::check_dispatch_args(c, h->rows_alloc, x, topk_weights, recv_x,
                                                   recv_sf, recv_topk_weights, recv_topk_idx);
      st != EP_OK)
    return st;
  if (const ep_status st = ep::check_device(h); st != EP_OK) return st;
  const ep::DispatchParams p = ep::dispatch_params(h, x, topk_weights, recv_x, recv_sf,
                                                   recv_topk_weights, recv_topk_idx);
  if (h->rows_alloc == 0) return EP_OK;  // nothing lands anywhere
  const cudaError_t ce =
      ep::launch_dispatch(p, c.use_fp8, c.use_tma_aligned_col_major_sf, c.num_sms,
                          reinterpret_cast<cudaStream_t>(stream));
  return ep::cuda_status(ce);
}

ep_status ep_layout_dispatch(const ep_config *cfg, const void *topk_idx, const void *x,
                             const float *topk_weights, void *recv_x, float *recv_sf,
                             float *recv_topk_weights, int32_t *recv_topk_idx,
                             ep_stream_t stream, ep_handle **out_handle, ep_layout_info *info) {
  if (out_handle == nullptr || info == nullptr) return EP_ERR_INVALID_ARG;
  *out_handle = nullptr;
  if (cfg == nullptr) return EP_ERR_INVALID_ARG;
  if (cfg->do_cpu_sync) return EP_ERR_INVALID_ARG;  // receive buffers are sized in advance
  if (const ep_status st = ep_validate_config(cfg); st != EP_OK) return st;
  if (const ep_status st =
          ep::check_dispatch_args(*cfg, ep::upper_bound(*cfg).rows, x, topk_weights, recv_x,
                                  recv_sf, recv_topk_weights, recv_topk_idx);
      st != EP_OK)
    return st;
  ep::LayoutSetup L;
  if (const ep_status st = ep::layout_setup(cfg, topk_idx, stream, &L); st != EP_OK) return st;
  ep_handle *h = ep::make_handle(L, L.b.rows);
  ep::DispatchParams p = ep::dispatch_params(h, x, topk_weights, recv_x, recv_sf,
                                             recv_topk_weights, recv_topk_idx);
  const ep_config &c = L.c;
  int layout_kernels = 0;
  // x is an input of this call, so it was complete before the layout
  // started: the dispatch, launched right behind the layout, loads (and
  // quantises) its first source rows while the layout runs
  cudaError_t ce = ep::launch_layout(L.lp, L.s, &layout_kernels);
  p.early_x = 1;
  if (ce == cudaSuccess && h->rows_alloc > 0)
    ce = ep::launch_dispatch(p, c.use_fp8, c.use_tma_aligned_col_major_sf, c.num_sms, L.s);
  if (ce != cudaSuccess) {
    cudaFreeAsync(L.dmem, L.s);
    delete h;
    return ep::cuda_status(ce);
  }
  ep::fill_info(h, -1, -1, layout_kernels, info);
  *out_handle = h;
  return EP_OK;
}

ep_status ep_dispatch_fp8(ep_handle *h, const void *x_fp8, const float *x_sf,
                          int64_t x_sf_token_stride, int64_t x_sf_hidden_stride,
                          const float *topk_weights, void *recv_x, float *recv_sf,
                          float *recv_topk_weights, int32_t *recv_topk_idx, ep_stream_t stream) {
  if (h == nullptr) return EP_ERR_INVALID_ARG;
  const ep_config &c = h->cfg;
  if (!c.use_fp8) return EP_ERR_INVALID_ARG;  // the handle's receive layout must be FP8
  const int T = c.num_tokens;
  if (T > 0 && (x_fp8 == nullptr || !aligned(x_fp8, 16) || x_sf == nullptr || !aligned(x_sf, 4)))
    return EP_ERR_INVALID_ARG;
  if (x_sf_token_stride < 0 || x_sf_hidden_stride < 0) return EP_ERR_INVALID_ARG;
  if (x_sf_token_stride > (int64_t(1) << 40) || x_sf_hidden_stride > (int64_t(1) << 40))
    return EP_ERR_INVALID_ARG;
  if (h->rows_alloc > 0 && (recv_x == nullptr || !aligned(recv_x, 16) || recv_sf == nullptr ||
                            !aligned(recv_sf, 4)))
    return EP_ERR_INVALID_ARG;
  if (recv_topk_weights != nullptr &&
      ((T > 0 && topk_weights == nullptr) || !aligned(recv_topk_weights, 4)))
    return EP_ERR_INVALID_ARG;
  if (topk_weights != nullptr && !aligned(topk_weights, 4)) return EP_ERR_INVALID_ARG;
  if (recv_topk_idx != nullptr && (c.do_expand || !aligned(recv_topk_idx, 4)))
    return EP_ERR_INVALID_ARG;
  if (const ep_status st = ep::check_device(h); st != EP_OK) return st;
  ep::DispatchParams p = ep::dispatch_params(h, nullptr, topk_weights, recv_x, recv_sf,
                                             recv_topk_weights, recv_topk_idx);
  p.xq = static_cast<const uint8_t *>(x_fp8);
  p.xs = x_sf;
  p.xs_ts = x_sf_token_stride;
  p.xs_hs = x_sf_hidden_stride;
  p.sf_src = x_sf;
  p.sf_src_ts = x_sf_token_stride;
  p.sf_src_hs = x_sf_hidden_stride;
  if (h->rows_alloc == 0) return EP_OK;
  const cudaError_t ce = ep::launch_dispatch(p, 2, c.use_tma_aligned_col_major_sf, c.num_sms,
                                             reinterpret_cast<cudaStream_t>(stream));
  return ep::cuda_status(ce);
}

ep_status ep_combine(const ep_handle *h, const void *y, const float *topk_weights,
                     const void *bias_0, const void *bias_1, const void *expert_bias, void *out,
                     ep_stream_t stream) {
  if (h == nullptr) return EP_ERR_INVALID_ARG;
  const ep_config &c = h->cfg;
  const int T = c.num_tokens;
  if (T > 0 && (out == nullptr || !aligned(out, 16))) return EP_ERR_INVALID_ARG;
  if (h->rows_alloc > 0 && (y == nullptr || !aligned(y, 16))) return EP_ERR_INVALID_ARG;
  if (topk_weights != nullptr && !aligned(topk_weights, 4)) return EP_ERR_INVALID_ARG;
  if ((bias_0 != nullptr && !aligned(bias_0, 16)) || (bias_1 != nullptr && !aligned(bias_1, 16)) ||
      (expert_bias != nullptr && !aligned(expert_bias, 16)))
    return EP_ERR_INVALID_ARG;
  if (const ep_status st = ep::check_device(h); st != EP_OK) return st;
  const ep::CombineParams p =
      ep::combine_params(h, y, topk_weights, bias_0, bias_1, expert_bias, out);
  const cudaError_t ce = ep::launch_combine(p, c.num_sms, reinterpret_cast<cudaStream_t>(stream));
  return ep::cuda_status(ce);
}

ep_status ep_dispatch_backward(const ep_handle *h, const void *grad_recv_x,
                               const float *grad_recv_topk_weights, void *grad_x,
                               float *grad_topk_weights, ep_stream_t stream) {
  if (h == nullptr) return EP_ERR_INVALID_ARG;
  const ep_config &c = h->cfg;
  const int T = c.num_tokens;
  if (T > 0 && (grad_x == nullptr || !aligned(grad_x, 16))) return EP_ERR_INVALID_ARG;
  if (h->rows_alloc > 0 && (grad_recv_x == nullptr || !aligned(grad_recv_x, 16)))
    return EP_ERR_INVALID_ARG;
  // grad_topk_weights asks for the weight reduction; its input may be absent
  // only when no row exists to hold it (rows_alloc == 0: every result is 0)
  if (grad_topk_weights == nullptr && grad_recv_topk_weights != nullptr) return EP_ERR_INVALID_ARG;
  if (grad_topk_weights != nullptr &&
      (!aligned(grad_topk_weights, 4) ||
       (h->rows_alloc > 0 &&
        (grad_recv_topk_weights == nullptr || !aligned(grad_recv_topk_weights, 4)))))
    return EP_ERR_INVALID_ARG;
  if (const ep_status st = ep::check_device(h); st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const ep::CombineParams p =
      ep::combine_params(h, grad_recv_x, nullptr, nullptr, nullptr, nullptr, grad_x);
  cudaError_t ce = ep::launch_combine(p, c.num_sms, s);
  if (ce == cudaSuccess && grad_topk_weights != nullptr) {
    ep::CombineWeightsParams q{};
    q.dst = h->lp.dst;
    q.g = grad_recv_topk_weights;
    q.out = grad_topk_weights;
    q.T = T;
    q.K = c.num_topk;
    q.do_expand = c.do_expand;
    ce = ep::launch_combine_weights(q, s);
  }
  return ep::cuda_status(ce);
}

ep_status ep_combine_backward(ep_handle *h, const void *grad_combined_x, void *grad_recv_x,
                              ep_stream_t stream) {
  if (h == nullptr) return EP_ERR_INVALID_ARG;
  const ep_config &c = h->cfg;
  if (c.num_tokens > 0 && (grad_combined_x == nullptr || !aligned(grad_combined_x, 16)))
    return EP_ERR_INVALID_ARG;
  if (h->rows_alloc > 0 && (grad_recv_x == nullptr || !aligned(grad_recv_x, 16)))
    return EP_ERR_INVALID_ARG;
  if (const ep_status st = ep::check_device(h); st != EP_OK) return st;
  const ep::DispatchParams p =
      ep::dispatch_params(h, grad_combined_x, nullptr, grad_recv_x, nullptr, nullptr, nullptr);
  if (h->rows_alloc == 0) return EP_OK;
  // always the BF16 copy, whatever the forward dispatch quantised to
  const cudaError_t ce = ep::launch_dispatch(p, 0, 0, c.num_sms, reinterpret_cast<cudaStream_t>(stream));
  return ep::cuda_status(ce);
}

void ep_handle_free(ep_handle *h) {
  if (h == nullptr) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != h->device) cudaSetDevice(h->device);
  if (cudaFreeAsync(h->dmem, h->stream) != cudaSuccess) {
    cudaGetLastError();  // e.g. the layout stream was destroyed: free synchronously
    cudaFree(h->dmem);
  }
  if (cur >= 0 && cur != h->device) cudaSetDevice(cur);
  delete h;
}

}  // extern "C"
