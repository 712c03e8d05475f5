// Internal declarations shared by the translation units of libep.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep.h"

namespace ep {

constexpr int kFp8Block = 128;          // 1x128 scale blocks
constexpr int kLayoutThreads = 1024;     // assign kernel CTA
constexpr int kLayoutChunkTokens = 256;  // tokens per layout chunk (<= 8192 slots with K <= 32)
// Rank layouts of at most this many chunks run as one kernel whose grid is a
// single thread-block cluster of one CTA per chunk plus one (above 8 CTAs: a
// non-portable cluster size, at most 16), if its shared memory fits
// kLayoutClusterSmem and the device can place it.
constexpr int kLayoutClusterChunks = 15;
constexpr size_t kLayoutClusterSmem = 96 * 1024;

// Control words at the head of the handle's device block.
enum CtrlSlot { kCtrlError = 0, kCtrlNumRecv = 2, kCtrlNumExpanded = 3, kCtrlWords = 8 };
// Handle words shared by dispatch launches: [0, 2) scale-gather handshake,
// [2, 5) dynamic scheduling (tokens handed out, CTAs finished, padding items).
constexpr int kDispSyncWords = 5;

// Pinned, device-mapped host words the count wait polls (do_cpu_sync).
// Mapped host words of the count wait.  Each word is (seq << 32 | value):
// it is current once its high half equals the call's sequence number, so the
// device needs no fence to order them and the host reads each word whole
// (aligned 8-byte accesses are single-copy atomic).
struct HostSync {
  volatile uint64_t num_recv;
  volatile uint64_t num_expanded;
  volatile uint64_t error;
  uint64_t pad[5];
};

// Everything a layout kernel needs; passed by value.
struct LayoutParams {
  const void *topk_idx;   // caller's [T, K]
  int idx_is_int64;
  int T, K, E, R, L, M, A;
  int do_expand;
  int fixed_cap;          // > 0: fixed-capacity layout, rows per expert (do_expand only)
  int32_t *disp_sync;     // [kDispSyncWords] handle only (else nullptr): dispatch
                          // scheduling and scale-gather handshake counters, zeroed
                          // by the layout
  int num_blocks;         // layout grid (one CTA per chunk of tokens)
  int blocks_per_src;     // chunks per source rank
  int src_ranks;          // source ranks holding tokens: ceil(T / M)
  int chunk_tokens;       // tokens per chunk
  int rank_warps;         // warps that rank slots in the assign kernel
  int64_t row_limit;      // rows at or past this are dropped (overflow)
  int32_t *topk32;        // [T, K]
  int32_t *dst;           // [T, K]
  int32_t *meta;          // [row_limit, 2]
  uint8_t *in_rank;       // [T, R]
  int32_t *cnt_e, *cnt_e_al, *psum_e;   // [E], [E], [E+1]
  int32_t *psum_pad;      // [E+1] exclusive prefix of the padding rows per expert
  int32_t *cnt_r, *psum_r, *psum_rs;    // [R], [R+1], [R, R+1]
  int32_t *ctrl;          // kCtrl* words
  int32_t *blk_e;         // [num_blocks, E] per-chunk expert counts
  int32_t *blk_r;         // [num_blocks, R] per-chunk rank counts
  unsigned *blk_err;      // [num_blocks] per-chunk EP_ERRBIT_* bits
  HostSync *host;         // device view of the mapped host words, or nullptr
  int32_t seq;            // value the count wait looks for
};

struct DispatchParams {
  const uint16_t *x;      // [T, H] bf16 bits
  const float *topk_w;    // [T, K] or nullptr
  const int32_t *topk32;  // [T, K]
  const int32_t *dst;     // [T, K]
  const int32_t *psum_e;  // [E+1]
  const int32_t *cnt_e;   // [E]
  const int32_t *psum_pad;  // [E+1] padding rows before expert e
  int T, K, E, L, H;
  int do_expand, zero_padding;
  int64_t max_pad_items;  // upper bound on padding work items (grid sizing only)
  int64_t rows_alloc;     // rows of recv_*
  int64_t sf_hidden_stride, sf_token_stride;
  void *recv_x;
  float *recv_sf;
  float *recv_w;
  int32_t *recv_idx;
  unsigned *err;          // the handle's error word (EP_ERRBIT_TIMEOUT)
  float *tok_scale;       // [T, H/128] FP8 scales per source token (handle scratch)
  const int32_t *meta;    // [rows, 2] recv_src_metadata
  const int32_t *num_rows;  // device total rows of the layout
  // pre-quantised input: e4m3 bytes [T, H] and scales x_sf[t * xs_ts + j * xs_hs]
  const uint8_t *xq;
  const float *xs;
  int64_t xs_ts, xs_hs;
  // per-token scales read by the column-major scale gather (element (t, j) at
  // sf_src[t * sf_src_ts + j * sf_src_hs]); sf_src_vec4 is set by the launcher
  const float *sf_src;
  int64_t sf_src_ts, sf_src_hs;
  int sf_src_vec4;
  // fixed-capacity layout: rows per expert (0 otherwise) and the scale stride
  // between experts' column-major slabs
  int fixed_cap;
  int64_t sf_expert_stride;
  // Quantising dispatch with column-major scales: every dispatch CTA adds 1 to
  // sf_sync[0] once its tokens' scales are written; the scale gather, launched
  // early, waits (bounded) for sf_sync_target and its last CTA resets both
  // counters.  sf_wait selects what the gather waits for (none / this
  // handshake / the whole dispatch grid).
  int32_t *sf_sync;
  int sf_sync_target;
  int sf_wait;
  // [3] dynamic scheduling: tokens past the first wave handed out, CTAs
  // finished, padding items handed out (the last CTA resets all three for
  // the next dispatch on the handle)
  int32_t *sched;
  // 1: x was complete before the kernel launched just ahead of this one
  // started (the layout of the same call), so the first rows of every CTA
  // are loaded and quantised before griddepcontrol.wait
  int early_x;
};

struct CombineParams {
  const uint16_t *y;      // [rows_alloc, H]
  const float *topk_w;    // [T, K] or nullptr
  const int32_t *topk32;  // [T, K]
  const int32_t *dst;     // [T, K]
  const uint16_t *bias0, *bias1;  // [T, H] or nullptr
  const uint16_t *ebias;  // [E, H] or nullptr
  uint16_t *out;          // [T, H]
  unsigned *err;          // the handle's error word (EP_ERRBIT_TIMEOUT)
  int T, K, H;
  int64_t rows_alloc;
};

struct CombineWeightsParams {
  const int32_t *dst;     // [T, K]
  const float *g;         // [rows_alloc] (expanded) or [rows_alloc, K] (rank layout)
  float *out;             // [T, K]
  int T, K;
  int do_expand;
};

// Dynamic shared memory above which a kernel must opt in with
// cudaFuncAttributeMaxDynamicSharedMemorySize: the 48 KB default window less
// a margin for the kernels' static shared memory (all below 8 KB).
constexpr size_t kDynSmemOptIn = 40 * 1024;

// Launchers (return the first CUDA error, cudaSuccess otherwise).
// launch_layout sets *kernels to the number of kernels it launched.
cudaError_t launch_layout(const LayoutParams &p, cudaStream_t s, int *kernels);
size_t layout_assign_smem(const LayoutParams &p);
int layout_rank_warps(int nkey);
// mode: 0 BF16 copy, 1 quantise BF16 to e4m3 + scales, 2 copy a pre-quantised input
cudaError_t launch_dispatch(const DispatchParams &p, int mode, int col_major,
                            int sm_cap, cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, int sm_cap, cudaStream_t s);
cudaError_t launch_combine_weights(const CombineWeightsParams &p, cudaStream_t s);

// Device facts, cached per device.
int device_sm_count(int device);

// Resident CTAs per SM of `func` at (threads, dynamic shared memory) on the
// current device, with the dynamic shared-memory opt-in (above
// kDynSmemOptIn) applied first.  Both are looked up once per device,
// function and shape and cached for the life of the process, so a launch
// makes no runtime query after the first of its shape.  per_sm = nullptr
// applies the opt-in only.
cudaError_t launch_geometry(const void *func, int threads, size_t smem, int *device,
                            int *per_sm);

}  // namespace ep
