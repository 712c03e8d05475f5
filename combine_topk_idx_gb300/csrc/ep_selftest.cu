// Self-test of the bounded device wait used by the TMA pipelines.
#include "ep_internal.cuh"
#include "ep_ptx.cuh"

namespace {

__device__ unsigned g_selftest_err;

__global__ void selftest_wait_kernel(int iters, uint32_t hint_ns, int signal) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ep::mbar_init(&bar, 1);
    ep::fence_mbar_init();
  }
  __syncthreads();
  if (signal && threadIdx.x == 0) ep::mbar_arrive(&bar);
  const bool ok = ep::mbar_wait_bounded(&bar, 0, iters, hint_ns);
  if (!ok && threadIdx.x == 0) atomicOr(&g_selftest_err, EP_ERRBIT_TIMEOUT);
}

}  // namespace

extern "C" ep_status ep_selftest_bounded_wait(int32_t wait_us, int32_t signal,
                                              uint32_t *error_bits, ep_stream_t stream) {
  if (error_bits == nullptr || wait_us < 1 || wait_us > 10 * 1000 * 1000) return EP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned zero = 0;
  if (cudaMemcpyToSymbolAsync(g_selftest_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return EP_ERR_CUDA;
  // attempts of at most 1 us each
  selftest_wait_kernel<<<1, 32, 0, s>>>(wait_us, 1000u, signal ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpyFromSymbolAsync(&bits, g_selftest_err, sizeof(bits), 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return EP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return EP_ERR_CUDA;
  *error_bits = bits;
  return EP_OK;
}
