// Allocation-free variant of the routing layout (ep_layout_noalloc).
//
// Some callers cannot allocate device memory at the point where they need
// the layout: a CUDA-graph capture that must stay free of allocation nodes,
// runtimes that hand out every byte of device memory themselves, or hosts
// whose allocator must not be entered from that thread.  This entry point
// runs the same two layout kernels as ep_layout (no host count wait) on
// caller-provided output buffers; the only scratch, the per-chunk expert /
// rank histograms, lives in a static device array instead of the handle.
#include <algorithm>
#include <mutex>
#include <vector>

#include "ep_internal.cuh"

namespace {

// Per-chunk histograms of every call: [chunks, E], then [chunks, R], then
// [chunks] error bits.  Held by every GPU that loads the library.
static __device__ __align__(256) int32_t g_layout_scratch[EP_NOALLOC_SCRATCH_WORDS];

// Device address of g_layout_scratch on `device` (current).  Looked up again
// on every call made outside a stream capture, so a context re-created after
// cudaDeviceReset gets its own address; inside a capture the address from
// the last call outside one is used (the first call on a device must
// therefore come before any capture).
ep_status scratch_address(int device, bool capturing, int32_t **out) {
  static std::mutex mu;
  static std::vector<int32_t *> addr;
  std::lock_guard<std::mutex> g(mu);
  if ((int)addr.size() <= device) addr.resize(device + 1, nullptr);
  if (addr[device] == nullptr || !capturing) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_layout_scratch);
    if (e != cudaSuccess || ptr == nullptr) return EP_ERR_CUDA;
    addr[device] = static_cast<int32_t *>(ptr);
  }
  *out = addr[device];
  return EP_OK;
}

}  // namespace

extern "C" ep_status ep_layout_noalloc(const ep_config *cfg, const void *topk_idx,
                                       const ep_layout_buffers *out, ep_stream_t stream) {
  ep_status st = ep_validate_config(cfg);
  if (st != EP_OK) return st;
  if (out == nullptr || cfg->do_cpu_sync) return EP_ERR_INVALID_ARG;
  const ep_config &c = *cfg;
  const int T = c.num_tokens, K = c.num_topk, E = c.num_experts, R = c.num_ranks;
  if (T > 0 && (topk_idx == nullptr ||
                reinterpret_cast<uintptr_t>(topk_idx) % (c.topk_idx_is_int64 ? 8 : 4) != 0))
    return EP_ERR_INVALID_ARG;
  int64_t rows = 0;
  st = ep_upper_bound_rows(cfg, &rows);
  if (st != EP_OK) return st;
  if (out->cnt_expert == nullptr || out->cnt_expert_aligned == nullptr ||
      out->psum_expert == nullptr || out->psum_padding == nullptr || out->cnt_rank == nullptr ||
      out->psum_rank == nullptr || out->psum_rank_src == nullptr || out->status == nullptr ||
      (T > 0 && (out->topk_idx32 == nullptr || out->dst_buffer_slot_idx == nullptr ||
                 out->is_token_in_rank == nullptr)) ||
      (rows > 0 && out->recv_src_metadata == nullptr))
    return EP_ERR_INVALID_ARG;
  // 8-byte rows of metadata and 4-byte packed rank rows are written whole
  if (reinterpret_cast<uintptr_t>(out->recv_src_metadata) % 8 != 0 ||
      reinterpret_cast<uintptr_t>(out->is_token_in_rank) % 4 != 0)
    return EP_ERR_INVALID_ARG;

  ep::LayoutParams lp{};
  lp.topk_idx = topk_idx;
  lp.idx_is_int64 = c.topk_idx_is_int64;
  lp.T = T; lp.K = K; lp.E = E; lp.R = R; lp.L = E / R;
  lp.M = c.num_max_tokens_per_rank;
  lp.A = c.expert_alignment;
  lp.do_expand = c.do_expand;
  lp.fixed_cap = c.fixed_capacity ? c.num_max_tokens_per_rank * c.num_ranks : 0;
  lp.row_limit = rows;
  lp.chunk_tokens = ep::kLayoutChunkTokens;
  const int64_t src_ranks = ((int64_t)T + lp.M - 1) / lp.M;
  const int64_t max_tok = std::min<int64_t>(lp.M, T);
  lp.blocks_per_src = (int)std::max<int64_t>(1, (max_tok + lp.chunk_tokens - 1) / lp.chunk_tokens);
  const int64_t chunks = std::max<int64_t>(1, src_ranks * lp.blocks_per_src);
  lp.src_ranks = (int)src_ranks;
  const int64_t words = chunks * ((int64_t)E + R + 1);
  if (words > EP_NOALLOC_SCRATCH_WORDS) return EP_ERR_UNSUPPORTED;
  lp.num_blocks = (int)chunks;
  lp.rank_warps = ep::layout_rank_warps(c.do_expand ? E : R);
  if (ep::layout_assign_smem(lp) > 220 * 1024) return EP_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess)
    return EP_ERR_CUDA;
  int32_t *scratch = nullptr;
  st = scratch_address(dev, cs != cudaStreamCaptureStatusNone, &scratch);
  if (st != EP_OK) return st;
  lp.blk_e = scratch;
  lp.blk_r = scratch + chunks * E;
  lp.blk_err = reinterpret_cast<unsigned *>(scratch + chunks * ((int64_t)E + R));
  lp.topk32 = out->topk_idx32;
  lp.dst = out->dst_buffer_slot_idx;
  lp.meta = out->recv_src_metadata;
  lp.in_rank = out->is_token_in_rank;
  lp.cnt_e = out->cnt_expert;
  lp.cnt_e_al = out->cnt_expert_aligned;
  lp.psum_e = out->psum_expert;
  lp.psum_pad = out->psum_padding;
  lp.cnt_r = out->cnt_rank;
  lp.psum_r = out->psum_rank;
  lp.psum_rs = out->psum_rank_src;
  lp.ctrl = out->status;
  lp.host = nullptr;
  int kernels = 0;
  const cudaError_t ce =
      ep::launch_layout(lp, reinterpret_cast<cudaStream_t>(stream), &kernels);
  return ce == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
