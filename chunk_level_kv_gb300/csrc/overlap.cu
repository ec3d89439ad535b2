// Adjacent-layer overlap of kept index lists (ChunkKV §4.2, the observation
// behind Algorithm 2: the indices selected in consecutive layers are highly
// similar by Jaccard similarity).
//
// One CTA per (sequence, KV head, adjacent pair l, l+1): list l is marked in a
// shared-memory bitmap of the sequence's T positions, list l+1 is probed
// against it, and the CTA writes |I_l ∩ I_{l+1}| and |I_l ∪ I_{l+1}|
// (= |I_l| + |I_{l+1}| - |I_l ∩ I_{l+1}|, the lists holding distinct positions).
// Positions outside [0, T) are ignored and counts are clamped to the list
// capacity, so a malformed list cannot write outside the bitmap.
#include "common.cuh"

namespace chunkkv {

constexpr int kOverlapThreads = 512;

__global__ void __launch_bounds__(kOverlapThreads)
overlap_kernel(const __grid_constant__ SeqTable st, int Hkv, int n_cap, const int32_t* __restrict__ indices,
               const int32_t* __restrict__ counts, int32_t* __restrict__ inter, int32_t* __restrict__ uni) {
  extern __shared__ uint32_t bitmap[];
  __shared__ int32_t warp_hits[kOverlapThreads / 32];
  const int nbh = st.B * Hkv;
  const int bh = blockIdx.x, l = blockIdx.y;
  const int b = bh / Hkv;
  const int T = st.cu[b + 1] - st.cu[b];
  const int words = (T + 31) >> 5;
  for (int i = threadIdx.x; i < words; i += blockDim.x) bitmap[i] = 0u;
  pdl_wait();
  const int64_t base_a = (int64_t)l * nbh + bh, base_b = base_a + nbh;
  const int ca = min(max(counts[base_a], 0), n_cap);
  const int cb = min(max(counts[base_b], 0), n_cap);
  const int32_t* ia = indices + base_a * n_cap;
  const int32_t* ib = indices + base_b * n_cap;
  __syncthreads();
  for (int i = threadIdx.x; i < ca; i += blockDim.x) {
    const int j = ia[i];
    if (j >= 0 && j < T) atomicOr(&bitmap[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  int hits = 0;
  for (int i = threadIdx.x; i < cb; i += blockDim.x) {
    const int j = ib[i];
    if (j >= 0 && j < T) hits += (bitmap[j >> 5] >> (j & 31)) & 1u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) hits += __shfl_xor_sync(0xffffffffu, hits, o);
  if ((threadIdx.x & 31) == 0) warp_hits[threadIdx.x >> 5] = hits;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < kOverlapThreads / 32; ++w) total += warp_hits[w];
    inter[base_a] = total;
    uni[base_a] = ca + cb - total;
  }
  pdl_trigger();
}

cudaError_t launch_overlap(const SeqTable& st, int Hkv, int n_cap, int n_lists, int max_T, const int32_t* indices,
                           const int32_t* counts, int32_t* inter, int32_t* uni, cudaStream_t s) {
  if (n_lists < 2 || st.B * Hkv == 0) return cudaSuccess;
  const size_t smem = (size_t)((max_T + 31) / 32) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(overlap_kernel, dim3(st.B * Hkv, n_lists - 1), dim3(kOverlapThreads), smem, s, st, Hkv, n_cap,
                    indices, counts, inter, uni);
}

}  // namespace chunkkv
