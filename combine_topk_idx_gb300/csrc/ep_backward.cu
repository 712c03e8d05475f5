// Weight-gradient reduction of dispatch_backward.
//
// DeepEP README, "Interfaces and examples": the backward of dispatch is a
// combine of the received gradients that also reduces the received top-k
// weights back to token order.  The data part runs in the combine kernel
// (unweighted mode: a token's distinct rows summed once each).  This kernel
// does the weights: per token, the fp32 sum of its distinct destination
// rows' weight entries, taken in the order the rows first appear in its
// slots.  Expanded layout: one scalar per row and one row per slot, so slot
// k reads its own row.  Rank layout: [rows, K] per row, and every column of
// the token's result sums that column over the token's rows.
//
// The work is T*K scalars against a [T, K] routing table; one thread per
// output element, the token's routing row read through L1.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kWeightThreads = 256;

__global__ void __launch_bounds__(kWeightThreads)
    combine_weights_kernel(CombineWeightsParams p) {
  const int64_t i = (int64_t)blockIdx.x * kWeightThreads + threadIdx.x;
  const int64_t n = (int64_t)p.T * p.K;
  if (i >= n) return;
  const int64_t t = i / p.K;
  const int c = (int)(i - t * p.K);
  const int32_t *d = p.dst + t * p.K;
  float acc = 0.0f;
  if (p.do_expand) {
    const int32_t r = __ldg(d + c);
    if (r >= 0) acc = __ldg(p.g + r);
  } else {
    for (int k = 0; k < p.K; ++k) {
      const int32_t r = __ldg(d + k);
      if (r < 0) continue;
      bool seen = false;
      for (int kp = 0; kp < k; ++kp) seen |= (__ldg(d + kp) == r);
      if (!seen) acc = __fadd_rn(acc, __ldg(p.g + (int64_t)r * p.K + c));
    }
  }
  p.out[i] = acc;
}

}  // namespace

cudaError_t launch_combine_weights(const CombineWeightsParams &p, cudaStream_t s) {
  const int64_t n = (int64_t)p.T * p.K;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + kWeightThreads - 1) / kWeightThreads;
  combine_weights_kernel<<<(unsigned)blocks, kWeightThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ep
