// Throughput probe of the exponential unit (a measurement aid, no counterpart in
// the ChunkKV notes).
//
// The window-scoring kernels evaluate one base-2 exponential (ex2.approx.ftz.f32,
// a MUFU instruction) per logit, so besides the HBM and tensor-core roofs the
// scoring phase has an exponential-unit roof: the number of logits divided by the
// rate at which the GPU can evaluate that instruction.  This kernel measures the
// rate: every thread runs CHUNKKV_PROBE_CHAINS independent chains of the same
// instruction, x <- 2^(-x), which stays in [0.5, 1] and never overflows, with
// enough warps per SM to keep the unit busy.  The caller times the launch.
#include "common.cuh"

namespace chunkkv {

__global__ void __launch_bounds__(CHUNKKV_PROBE_THREADS)
ex2_probe_kernel(float* __restrict__ sink, int iters) {
  float x[CHUNKKV_PROBE_CHAINS];
#pragma unroll
  for (int i = 0; i < CHUNKKV_PROBE_CHAINS; ++i) x[i] = 0.5f + 1e-7f * (float)(threadIdx.x * CHUNKKV_PROBE_CHAINS + i);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < CHUNKKV_PROBE_CHAINS; ++i) {
      float y;
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-x[i]));
      x[i] = y;
    }
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < CHUNKKV_PROBE_CHAINS; ++i) s += x[i];
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace chunkkv

extern "C" chunkkv_status chunkkv_probe_ex2(float* sink, int32_t blocks, int32_t iters, chunkkv_stream_t stream) {
  if (sink == nullptr || blocks < 1 || iters < 1) return CHUNKKV_ERR_INVALID_ARG;
  chunkkv::ex2_probe_kernel<<<blocks, CHUNKKV_PROBE_THREADS, 0, (cudaStream_t)stream>>>(sink, iters);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return CHUNKKV_ERR_CUDA;
  chunkkv::g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return CHUNKKV_OK;
}
