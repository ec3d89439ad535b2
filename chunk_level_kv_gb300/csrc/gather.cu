// K/V gather by a kept-index list (ChunkKV §4.1 Algorithm 1 step 6,
// index_select), batched over the layers that share one list (§4.2
// Algorithm 2) and over ragged sequences.
//
// Pure HBM traffic: every kept row is read once from K and V and written once
// to K' and V'.  Rows are moved as 16-byte vectors; the CTAs of one (layer,
// sequence, head) cover its output rows in order, so the writes are fully
// coalesced and each 256-byte key row (bf16, d = 128) is one coalesced read.
// Rows at or beyond counts[b][h] are skipped.
#include "common.cuh"

namespace chunkkv {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// grid.y = layer * (B * Hkv) + (b * Hkv + h); grid.x covers n_cap * vpr vectors.
__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(GatherGeom gg, const __grid_constant__ SeqTable st, const __grid_constant__ GatherArgs ga,
              const int32_t* __restrict__ indices, const int32_t* __restrict__ counts) {
  const int nbh = st.B * gg.Hkv;
  const int y = blockIdx.y;
  const int layer = y / nbh;
  const int bh = y - layer * nbh;
  const int b = bh / gg.Hkv, h = bh - b * gg.Hkv;
  if (gg.pair && !(b & 1)) return;                       // a kept prefix: nothing to append
  const int obh = gg.pair ? (b >> 1) * gg.Hkv + h : bh;  // its list and output rows
  const int grp = (gg.l0 + layer) / gg.n_reuse;          // the index list this layer uses
  indices += grp * gg.idx_gs;
  counts += grp * gg.cnt_gs;
  pdl_wait();
  const int cnt = min(max(counts[obh], 0), gg.n_cap);    // never beyond the output rows
  const int T = st.cu[b + 1] - st.cu[b];
  const int vpr_shift = __ffs(gg.d * gg.elt / 16) - 1;        // vectors per row (a power of two)
  const int vpr = 1 << vpr_shift;
  const int total = T > 0 ? cnt << vpr_shift : 0;
  const int32_t* idx = indices + (int64_t)obh * gg.n_cap;
  const char* kl = (const char*)ga.k[layer];
  const char* vl = (const char*)ga.v[layer];
  const int64_t row_stride = gg.kv_stride_t * gg.elt;
  const int64_t head_off = ((int64_t)st.cu[b] * gg.kv_stride_t + (int64_t)h * gg.kv_stride_h) * gg.elt;
  uint4* ko = (uint4*)((char*)ga.ko[layer] + (int64_t)obh * gg.n_cap * gg.d * gg.elt);
  uint4* vo = (uint4*)((char*)ga.vo[layer] + (int64_t)obh * gg.n_cap * gg.d * gg.elt);

  const int step = gridDim.x * blockDim.x;
  for (int base = blockIdx.x * blockDim.x * kGatherUnroll + threadIdx.x; base < total;
       base += step * kGatherUnroll) {
    uint4 kv[kGatherUnroll], vv[kGatherUnroll];
#pragma unroll
    for (int i = 0; i < kGatherUnroll; ++i) {
      const int slot = base + i * blockDim.x;
      if (slot < total) {
        const int r = slot >> vpr_shift, vi = slot & (vpr - 1);
        const int j = min(max(idx[r], 0), T - 1);             // indices are in [0, T) by contract
        const int64_t off = head_off + (int64_t)j * row_stride;
        kv[i] = ld_stream((const uint4*)(kl + off) + vi);
        vv[i] = ld_stream((const uint4*)(vl + off) + vi);
      }
    }
#pragma unroll
    for (int i = 0; i < kGatherUnroll; ++i) {
      const int slot = base + i * blockDim.x;
      if (slot < total) {
        st_stream(ko + slot, kv[i]);
        st_stream(vo + slot, vv[i]);
      }
    }
  }
  pdl_trigger();
}

// Portable variant for row sizes that are not a power-of-two number of vectors.
__global__ void __launch_bounds__(kGatherThreads)
gather_any_kernel(GatherGeom gg, const __grid_constant__ SeqTable st, const __grid_constant__ GatherArgs ga,
                  const int32_t* __restrict__ indices, const int32_t* __restrict__ counts) {
  const int nbh = st.B * gg.Hkv;
  const int layer = blockIdx.y / nbh;
  const int bh = blockIdx.y - layer * nbh;
  const int b = bh / gg.Hkv, h = bh - b * gg.Hkv;
  if (gg.pair && !(b & 1)) return;
  const int obh = gg.pair ? (b >> 1) * gg.Hkv + h : bh;
  const int grp = (gg.l0 + layer) / gg.n_reuse;
  indices += grp * gg.idx_gs;
  counts += grp * gg.cnt_gs;
  pdl_wait();
  const int vpr = gg.d * gg.elt / 16;
  const int T = st.cu[b + 1] - st.cu[b];
  const int total = T > 0 ? min(max(counts[obh], 0), gg.n_cap) * vpr : 0;
  const int32_t* idx = indices + (int64_t)obh * gg.n_cap;
  const int64_t head_off = ((int64_t)st.cu[b] * gg.kv_stride_t + (int64_t)h * gg.kv_stride_h) * gg.elt;
  uint4* ko = (uint4*)((char*)ga.ko[layer] + (int64_t)obh * gg.n_cap * gg.d * gg.elt);
  uint4* vo = (uint4*)((char*)ga.vo[layer] + (int64_t)obh * gg.n_cap * gg.d * gg.elt);
  for (int slot = blockIdx.x * blockDim.x + threadIdx.x; slot < total; slot += gridDim.x * blockDim.x) {
    const int r = slot / vpr, vi = slot - r * vpr;
    const int j = min(max(idx[r], 0), T - 1);
    const int64_t off = head_off + (int64_t)j * gg.kv_stride_t * gg.elt;
    ko[slot] = ld_stream((const uint4*)((const char*)ga.k[layer] + off) + vi);
    vo[slot] = ld_stream((const uint4*)((const char*)ga.v[layer] + off) + vi);
  }
  pdl_trigger();
}

cudaError_t launch_gather(const Plan& pl, const GatherGeom& gg, const SeqTable& st, const GatherArgs& ga,
                          const int32_t* indices, const int32_t* counts, cudaStream_t s) {
  const int nbh = pl.B * pl.Hkv;
  if (nbh == 0 || pl.n_cap == 0 || ga.n_layers == 0) return cudaSuccess;
  const int vpr = gg.d * gg.elt / 16;
  const int64_t slots = (int64_t)pl.n_cap * vpr;
  const bool pow2 = (vpr & (vpr - 1)) == 0;
  const int per_block = kGatherThreads * (pow2 ? kGatherUnroll : 1);
  int gx = (int)((slots + per_block - 1) / per_block);
  if (gx < 1) gx = 1;
  dim3 grid(gx, nbh * ga.n_layers);
  if (pow2) return launch_pdl(gather_kernel, grid, dim3(kGatherThreads), 0, s, gg, st, ga, indices, counts);
  return launch_pdl(gather_any_kernel, grid, dim3(kGatherThreads), 0, s, gg, st, ga, indices, counts);
}

}  // namespace chunkkv
