// Finalisation helpers shared by the finalisation kernels (score.cu, select.cu).
//
// Chunk i of a scoring unit scores A_i = sum_r bin[i][r] * 2^(R_r - lse_r)
// (ChunkKV §4.1 Algorithm 1 step 3 with the probabilities of Kara §2 Eq. (1)):
// bins and R come from a scoring kernel, lse_r is the row's base-2 log-sum-exp
// over every unit of its head.
#pragma once

#include "common.cuh"

namespace chunkkv {

// weight of one row: 2^(R - lse), zero for a row that saw no key in this unit
__device__ __forceinline__ float fin_weight(float R, float lse) { return R == -INFINITY ? 0.f : exp2f(R - lse); }

// Weights of rows r .. r+NV-1 (r a multiple of NV, NV in {1, 4, 8}).
template <bool LSE, int NV>
__device__ __forceinline__ void fin_weights(float (&wv)[NV], const float* wts, const float* Rrow, const float* Lrow,
                                            int r) {
  if constexpr (!LSE) {
#pragma unroll
    for (int j = 0; j < NV; j += (NV >= 4 ? 4 : 1)) {
      if constexpr (NV >= 4) {
        const float4 x = *reinterpret_cast<const float4*>(wts + r + j);
        wv[j] = x.x, wv[j + 1] = x.y, wv[j + 2] = x.z, wv[j + 3] = x.w;
      } else {
        wv[j] = wts[r + j];
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NV; j += (NV >= 4 ? 4 : 1)) {
      if constexpr (NV >= 4) {
        const float4 R = *reinterpret_cast<const float4*>(Rrow + r + j);
        const float4 L = *reinterpret_cast<const float4*>(Lrow + r + j);
        wv[j] = fin_weight(R.x, L.x), wv[j + 1] = fin_weight(R.y, L.y);
        wv[j + 2] = fin_weight(R.z, L.z), wv[j + 3] = fin_weight(R.w, L.w);
      } else {
        wv[j] = fin_weight(Rrow[r + j], Lrow[r + j]);
      }
    }
  }
}

// Base-2 log-sum-exp merge: (M, S), S relative to 2^M, absorbs the pair (Mv,
// Sv); an empty pair (Sv = 0: the row saw no key of that unit) adds nothing.
__device__ __forceinline__ void lse_merge(float& M, float& S, float Mv, float Sv) {
  if (Sv == 0.f) return;
  const float Mn = fmaxf(M, Mv);
  S = S * exp2f(M - Mn) + Sv * exp2f(Mv - Mn);
  M = Mn;
}

constexpr int kFinGroup = 8;                    // chunks one warp reduces at a time
constexpr int kFinWideGroup = 16;               // the same when one load per chunk covers a lane's rows

// w*G of at most 128 rows in fours: every lane's rows of a chunk are one 8-byte load, so a warp
// step takes kFinWideGroup chunks to keep as many bytes in flight as the wider row counts do.
__host__ __device__ __forceinline__ bool fin_wide(int wG) { return (wG & 3) == 0 && wG <= 128; }

// Warp sums of N values per lane (N a power of two, 2 <= N <= 32) in N - 1 + 5 - log2 N
// shuffles instead of 5 N: at each of the first log2 N levels a lane keeps half of its values
// and adds its partner's copies of them, trading the other half.  Returns the index of the sum
// the lane ends with, in v[0]: value (lane / (32 / N)), held by 32 / N lanes each.
template <int N>
__device__ __forceinline__ int warp_sum_each(float (&v)[N], int lane) {
  static_assert(N >= 2 && N <= 32 && (N & (N - 1)) == 0, "a power of two up to 32");
  int base = 0;
#pragma unroll
  for (int h = N / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;                   // keeps the upper half of its values
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float keep = upper ? v[i + h] : v[i];
      const float give = upper ? v[i] : v[i + h];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
    }
    base += upper ? h : 0;
  }
#pragma unroll
  for (int o = 16 / N; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  return base;
}

// One warp: the scores of chunks 0 .. m-1 (m <= kFinGroup) of a unit, whose bins
// start at cbase (chunk stride wG), into out[0 .. m-1].  Lanes take consecutive
// rows (coalesced bin loads), all loads of a step are issued together, and each
// lane forms the weights of its own rows (from R and lse when LSE, else read from
// wts); the rows are reduced with shuffles.
// KG: chunks of the step (kFinGroup, or kFinWideGroup when fin_wide(wG)).
template <bool LSE, int KG = kFinGroup>
__device__ __forceinline__ void fin_group(const bin_t* __restrict__ cbase, int wG, int m, const float* wts,
                                          const float* Rrow, const float* Lrow, float* out, int lane) {
  constexpr int kG = KG;
  float acc[kG];
#pragma unroll
  for (int i = 0; i < kG; ++i) acc[i] = 0.f;
  if (KG == kFinGroup && (wG & 7) == 0 && wG >= 256) {
    // eight consecutive rows per lane: 16-byte loads of eight bins, kG of them in flight
    for (int r = 8 * lane; r < wG; r += 256) {
      uint4 v[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i)
        v[i] = i < m ? __ldcs(reinterpret_cast<const uint4*>(cbase + (int64_t)i * wG + r)) : make_uint4(0u, 0u, 0u, 0u);
      float wv[8];
      fin_weights<LSE, 8>(wv, wts, Rrow, Lrow, r);
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const float2 b01 = bin_decode2(v[i].x), b23 = bin_decode2(v[i].y);
        const float2 b45 = bin_decode2(v[i].z), b67 = bin_decode2(v[i].w);
        acc[i] = fmaf(b01.x, wv[0], fmaf(b01.y, wv[1], fmaf(b23.x, wv[2], fmaf(b23.y, wv[3], acc[i]))));
        acc[i] = fmaf(b45.x, wv[4], fmaf(b45.y, wv[5], fmaf(b67.x, wv[6], fmaf(b67.y, wv[7], acc[i]))));
      }
    }
  } else if ((wG & 3) == 0) {
    // four consecutive rows per lane: 8-byte loads of four bins, kG of them in flight
    for (int r = 4 * lane; r < wG; r += 128) {
      uint2 v[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i)
        v[i] = i < m ? __ldcs(reinterpret_cast<const uint2*>(cbase + (int64_t)i * wG + r)) : make_uint2(0u, 0u);
      float wv[4];
      fin_weights<LSE, 4>(wv, wts, Rrow, Lrow, r);
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const float2 b01 = bin_decode2(v[i].x), b23 = bin_decode2(v[i].y);
        acc[i] = fmaf(b01.x, wv[0], fmaf(b01.y, wv[1], fmaf(b23.x, wv[2], fmaf(b23.y, wv[3], acc[i]))));
      }
    }
  } else {
    for (int r = lane; r < wG; r += 32) {
      float v[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i) v[i] = i < m ? bin_decode(__ldcs(cbase + (int64_t)i * wG + r)) : 0.f;
      float wv[1];
      fin_weights<LSE, 1>(wv, wts, Rrow, Lrow, r);
#pragma unroll
      for (int i = 0; i < kG; ++i) acc[i] = fmaf(v[i], wv[0], acc[i]);
    }
  }
  const int ch = warp_sum_each<kG>(acc, lane);
  if ((lane & (32 / kG - 1)) == 0 && ch < m) out[ch] = acc[0];
}

}  // namespace chunkkv
