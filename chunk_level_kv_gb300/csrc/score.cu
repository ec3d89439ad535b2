// Window scoring, portable SIMT path, and the per-unit finalisation shared by
// every scoring path.
//
// ChunkKV §4.1 Algorithm 1 steps 1-3 with the probabilities of Kara §2 Eq. (1):
//   A[b][h][i] = sum_{rows r of head h} sum_{j in chunk i} exp(s_rj - lse_r),
//   s_rj = <Q_w row r, K_j> / sqrt(d),  lse_r = log sum_{j < T_b} exp(s_rj).
//
// The keys of a (sequence, head) are split into units of `cpu` whole chunks.
// A scoring kernel writes, per unit and window row r,
//   R_r   a reference exponent (base 2: logits times log2(e)/sqrt(d)),
//   l_r   = sum_{j in unit} 2^(t_rj - R_r),
//   bin[i][r] = sum_{j in chunk i} 2^(t_rj - R_r)   for the unit's chunks,
// R and l in fp32, the bins as 16-bit unsigned floats (bin_encode).  lse_kernel
// then forms lse_r over every unit of the head, and finalize_kernel
// the weights 2^(R_r - lse_r) and A_i = sum_r bin[i][r] * weight_r.  This
// single pass over K needs no second read of the keys and no grid barrier.
#include "fin.cuh"

namespace chunkkv {

// ------------------------------------------------------------------ SIMT scoring
// One CTA per unit, one thread per window row (rows in blocks of kRows); K is
// staged through shared memory in tiles of kKeys keys.  The unit's row maximum
// is found in a first sweep so that the bins use the exact unit maximum as
// reference (the portable path trades a second dot product for simplicity).
constexpr int kSimtRows = 128;
constexpr int kSimtKeys = 32;

template <typename E>
__global__ void __launch_bounds__(kSimtRows)
score_simt_kernel(const E* __restrict__ q, const E* __restrict__ k, ScoreGeom g,
                  const __grid_constant__ SeqTable st, float* __restrict__ rl,
                  bin_t* __restrict__ bins) {
  extern __shared__ float smem[];
  const int ld = g.d + 1;                       // padded rows: conflict-free per-thread rows
  float* qs = smem;                             // [kSimtRows][ld]
  float* ks = smem + kSimtRows * ld;            // [kSimtKeys][ld]

  int b, h, u;
  const int gu = blockIdx.x;
  decode_unit(st, g.Hkv, gu, b, h, u);
  const int T = st.cu[b + 1] - st.cu[b];
  const int k0 = u * g.ku;
  const int nk = min(g.ku, T - k0);
  const E* kbase = k + (int64_t)(st.cu[b] + k0) * g.kv_stride_t + (int64_t)h * g.kv_stride_h;
  const int tid = threadIdx.x;
  pdl_wait();

  for (int rb = 0; rb < g.wG; rb += kSimtRows) {
    __syncthreads();
    for (int i = tid; i < kSimtRows * g.d; i += blockDim.x) {
      int row = i / g.d, e = i % g.d, r = rb + row;
      float val = 0.f;
      if (r < g.wG) {
        int gm = r / g.w, qi = r % g.w;           // row r = (group member gm, window row qi)
        val = to_float(q[(int64_t)(b >> g.pair) * g.q_stride_b + (int64_t)qi * g.q_stride_w +
                         (int64_t)(h * g.G + gm) * g.q_stride_h + e]);
      }
      qs[row * ld + e] = val;
    }
    const int r = rb + tid;
    const bool active = r < g.wG;
    const float* qrow = qs + tid * ld;
    // causal window: the row's window query (r mod w) sees keys up to T - w + (r mod w);
    // in unit-local key numbers that is `last` (may be negative: nothing visible)
    const int last = g.causal ? T - g.w + (g.w > 0 ? r % g.w : 0) - k0 : INT_MAX;

    // sweep 1: row maximum of the base-2 exponents over the unit
    float m = -INFINITY;
    for (int kt = 0; kt < nk; kt += kSimtKeys) {
      const int nt = min(kSimtKeys, nk - kt);
      __syncthreads();
      for (int i = tid; i < nt * g.d; i += blockDim.x) {
        int j = i / g.d, e = i % g.d;
        ks[j * ld + e] = to_float(kbase[(int64_t)(kt + j) * g.kv_stride_t + e]);
      }
      __syncthreads();
      if (active) {
        for (int j = 0; j < nt && kt + j <= last; ++j) {
          float dot = 0.f;
          const float* kr = ks + j * ld;
          for (int e = 0; e < g.d; ++e) dot = fmaf(qrow[e], kr[e], dot);
          m = fmaxf(m, dot * g.alpha);
        }
      }
    }
    // sweep 2: exponentials relative to the unit maximum, summed per chunk; the
    // reference is shifted by kBinShift, so the bins are formed in their scale
    m += kBinShift;
    float acc = 0.f, l = 0.f;
    int cur = 0;
    bin_t* brow = bins + (int64_t)gu * g.cpu * g.wG + r;
    for (int kt = 0; kt < nk; kt += kSimtKeys) {
      const int nt = min(kSimtKeys, nk - kt);
      __syncthreads();
      for (int i = tid; i < nt * g.d; i += blockDim.x) {
        int j = i / g.d, e = i % g.d;
        ks[j * ld + e] = to_float(kbase[(int64_t)(kt + j) * g.kv_stride_t + e]);
      }
      __syncthreads();
      if (active) {
        for (int j = 0; j < nt; ++j) {
          float dot = 0.f;
          const float* kr = ks + j * ld;
          for (int e = 0; e < g.d; ++e) dot = fmaf(qrow[e], kr[e], dot);
          const int ch = (kt + j) / g.c;
          if (ch != cur) {
            brow[(int64_t)cur * g.wG] = bin_encode_sat(acc);
            acc = 0.f;
            cur = ch;
          }
          const float p = kt + j <= last ? exp2f(dot * g.alpha - m) : 0.f;
          acc += p;
          l += p;
        }
      }
    }
    if (active) {
      brow[(int64_t)cur * g.wG] = bin_encode_sat(acc);
      rl[((int64_t)gu * 2 + 0) * g.wG + r] = m;
      rl[((int64_t)gu * 2 + 1) * g.wG + r] = l;
    }
  }
  pdl_trigger();
}

cudaError_t launch_score_simt(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* q,
                              const void* k, float* rl, bin_t* bins, cudaStream_t s) {
  if (g.n_units == 0 || g.wG == 0) return cudaSuccess;
  const size_t smem = (size_t)(kSimtRows + kSimtKeys) * (g.d + 1) * sizeof(float);
  cudaError_t e;
  if (pl.elt == 2) {
    e = cudaFuncSetAttribute(score_simt_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(score_simt_kernel<__nv_bfloat16>, dim3(g.n_units), dim3(kSimtRows), smem, s,
                   (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, g, st, rl, bins);
    if (e != cudaSuccess) return e;
  } else {
    e = cudaFuncSetAttribute(score_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(score_simt_kernel<float>, dim3(g.n_units), dim3(kSimtRows), smem, s, (const float*)q,
                   (const float*)k, g, st, rl, bins);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ finalisation
// One CTA per (unit, block of up to 128 chunks, reuse group).  Chunk i of the
// unit scores A_i = sum_r bin[i][r] * 2^(R_r - lse_r); each warp takes eight
// chunks at a time with its lanes on consecutive rows (coalesced bin loads).
//  - With an lse array (lse_kernel ran before), every lane forms the weights
//    of its own rows from R and lse as it loads its bins: all loads of a step
//    are issued together and the CTA needs no shared memory or barrier.
//  - Without one (the no-allocation scoring call), the weights go to shared
//    memory first, lse_r being formed from the (R, l) pairs of every unit of
//    the head.
constexpr int kFinThreads = 256;
constexpr int kFinChunks = 128;                 // chunks per CTA: blockIdx.y tiles a unit

// WG > 0: w*G known at compile time (bin addresses as immediates), else read from g.
template <bool LSE, int WG>
__global__ void __launch_bounds__(kFinThreads, 4)
finalize_kernel(ScoreGeom g, const __grid_constant__ SeqTable st, const float* __restrict__ rl,
                const bin_t* __restrict__ bins, const float* __restrict__ lse_rows, float* __restrict__ scores) {
  extern __shared__ float wts[];                // [wG], only without an lse array
  int b, h, u;
  const int gu = blockIdx.x;
  const int cb = blockIdx.y * kFinChunks;       // this CTA's block of the unit's chunks
  rl += blockIdx.z * g.rl_gs;                   // this CTA's reuse group
  bins += blockIdx.z * g.bins_gs;
  scores += blockIdx.z * g.scores_gs;
  pdl_wait();
  decode_unit(st, g.Hkv, gu, b, h, u);
  if (g.pair && !(b & 1)) return;               // a kept prefix: in the normaliser only
  const int T = st.cu[b + 1] - st.cu[b];
  const int C = (T + g.c - 1) / g.c;
  if (min(g.cpu, C - u * g.cpu) <= cb) return;  // no chunk of this unit in this block
  const float* Rrow = rl + (int64_t)gu * 2 * g.wG;                 // R of this unit's rows
  const float* Lrow = nullptr;
  if constexpr (LSE) {
    Lrow = lse_rows + blockIdx.z * g.lse_gs + ((int64_t)b * g.Hkv + h) * g.wG;
  } else {
    const int U = st.uoff[b + 1] - st.uoff[b];
    const int64_t stride_u = (int64_t)g.Hkv * 2 * g.wG;          // between units of one head
    const float* rl_head = rl + ((int64_t)st.uoff[b] * g.Hkv + h) * 2 * g.wG;
    for (int r = threadIdx.x; r < g.wG; r += blockDim.x) {
      float M = -INFINITY;
      for (int v = 0; v < U; ++v) M = fmaxf(M, rl_head[v * stride_u + r]);
      float S = 0.f;
      for (int v = 0; v < U; ++v) {
        const float l = rl_head[v * stride_u + g.wG + r];
        if (l > 0.f) S += l * exp2f(rl_head[v * stride_u + r] - M);   // units the row saw no key of add nothing
      }
      wts[r] = fin_weight(Rrow[r], M + log2f(S));
    }
    __syncthreads();
  }

  const int nc = min(min(g.cpu, C - u * g.cpu) - cb, kFinChunks);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wg = WG > 0 ? WG : g.wG;
  const bin_t* ub = bins + ((int64_t)gu * g.cpu + cb) * wg;
  float* out = scores + ((int64_t)(b >> g.pair) * g.Hkv + h) * g.C_max + (int64_t)u * g.cpu + cb;
  constexpr int kW = kFinThreads / 32;
  if (fin_wide(wg)) {
    for (int ch0 = warp * kFinWideGroup; ch0 < nc; ch0 += kW * kFinWideGroup)
      fin_group<LSE, kFinWideGroup>(ub + (int64_t)ch0 * wg, wg, min(kFinWideGroup, nc - ch0), wts, Rrow, Lrow,
                                    out + ch0, lane);
  } else {
    for (int ch0 = warp * kFinGroup; ch0 < nc; ch0 += kW * kFinGroup)
      fin_group<LSE>(ub + (int64_t)ch0 * wg, wg, min(kFinGroup, nc - ch0), wts, Rrow, Lrow, out + ch0, lane);
  }
  pdl_trigger();
}

// Row log-sum-exp (base 2) of every (sequence, head) from the per-unit (R, l)
// pairs: lse_r = M + log2(sum_u l_u 2^(R_u - M)), M = max_u R_u.  One CTA per
// (sequence, head, 32 rows): lane = row (128-byte loads), the 8 warps take every
// 8th unit, four units per step with their loads issued together, and the
// partial (M, S) pairs are merged through shared memory.
constexpr int kLseThreads = 256;

__global__ void __launch_bounds__(kLseThreads)
lse_kernel(ScoreGeom g, const __grid_constant__ SeqTable st, const float* __restrict__ rl,
           float* __restrict__ lse) {
  constexpr int W = kLseThreads / 32;
  __shared__ float shM[W][32], shS[W][32];
  const int bh = blockIdx.x;
  const int b = bh / g.Hkv, h = bh - b * g.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.y * 32 + lane;
  // paired sequences: the units of the kept prefix and of the tail (adjacent) merge into one row lse
  const int b0 = g.pair ? (b & ~1) : b, b1 = g.pair ? (b | 1) + 1 : b + 1;
  const int U = st.uoff[b1] - st.uoff[b0];
  rl += blockIdx.z * g.rl_gs;                   // this CTA's reuse group
  lse += blockIdx.z * g.lse_gs;
  pdl_wait();
  const int64_t ustride = (int64_t)g.Hkv * 2 * g.wG;
  const float* base = rl + ((int64_t)st.uoff[b0] * g.Hkv + h) * 2 * g.wG + r;
  float M = -INFINITY, S = 0.f;
  if (r < g.wG) {
    int v = warp;
    for (; v + 3 * W < U; v += 4 * W) {
      float Rv[4], lv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        Rv[i] = base[(v + i * W) * ustride];
        lv[i] = base[(v + i * W) * ustride + g.wG];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) lse_merge(M, S, Rv[i], lv[i]);
    }
    for (; v < U; v += W) lse_merge(M, S, base[v * ustride], base[v * ustride + g.wG]);
  }
  shM[warp][lane] = M;
  shS[warp][lane] = S;
  __syncthreads();
  if (warp == 0 && r < g.wG) {
    float Mt = -INFINITY, St = 0.f;
    for (int w2 = 0; w2 < W; ++w2) lse_merge(Mt, St, shM[w2][lane], shS[w2][lane]);
    lse[(int64_t)bh * g.wG + r] = Mt + log2f(St);
  }
  pdl_trigger();
}

// The same for heads of few units (kLseRowsMaxUnits at most): one thread per
// (sequence, head, row) merges all of the row's units, four loads in flight, and
// a CTA covers 128 rows; no warps split the units, since most would be idle.
constexpr int kLseRowsMaxUnits = 16;

__global__ void __launch_bounds__(128)
lse_rows_kernel(ScoreGeom g, const __grid_constant__ SeqTable st, const float* __restrict__ rl,
                float* __restrict__ lse) {
  const int bh = blockIdx.x;
  const int b = bh / g.Hkv, h = bh - b * g.Hkv;
  const int r = blockIdx.y * 128 + threadIdx.x;
  const int b0 = g.pair ? (b & ~1) : b, b1 = g.pair ? (b | 1) + 1 : b + 1;
  const int U = st.uoff[b1] - st.uoff[b0];
  rl += blockIdx.z * g.rl_gs;
  lse += blockIdx.z * g.lse_gs;
  pdl_wait();
  if (r < g.wG) {
    const int64_t ustride = (int64_t)g.Hkv * 2 * g.wG;
    const float* base = rl + ((int64_t)st.uoff[b0] * g.Hkv + h) * 2 * g.wG + r;
    float M = -INFINITY, S = 0.f;
    int v = 0;
    for (; v + 3 < U; v += 4) {
      float Rv[4], lv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        Rv[i] = base[(v + i) * ustride];
        lv[i] = base[(v + i) * ustride + g.wG];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) lse_merge(M, S, Rv[i], lv[i]);
    }
    for (; v < U; ++v) lse_merge(M, S, base[v * ustride], base[v * ustride + g.wG]);
    lse[(int64_t)bh * g.wG + r] = M + log2f(S);
  }
  pdl_trigger();
}

cudaError_t launch_lse(const ScoreGeom& g, const SeqTable& st, const float* rl, float* lse, int n_groups,
                       cudaStream_t s) {
  if (g.n_units == 0 || g.wG == 0 || n_groups == 0) return cudaSuccess;
  int u_max = 0;                                  // units of the longest (paired) sequence, per head
  for (int b = 0; b < st.B; b += g.pair ? 2 : 1) {
    const int b1 = g.pair ? std::min(b + 2, st.B) : b + 1;
    u_max = std::max(u_max, st.uoff[b1] - st.uoff[b]);
  }
  if (u_max <= kLseRowsMaxUnits) {
    dim3 grid(st.B * g.Hkv, (g.wG + 127) / 128, n_groups);
    return launch_pdl(lse_rows_kernel, grid, dim3(128), 0, s, g, st, rl, lse);
  }
  dim3 grid(st.B * g.Hkv, (g.wG + 31) / 32, n_groups);
  return launch_pdl(lse_kernel, grid, dim3(kLseThreads), 0, s, g, st, rl, lse);
}

// Scores of a head with no window rows are all zero (no attention mass).
__global__ void zero_scores_kernel(ScoreGeom g, const __grid_constant__ SeqTable st, float* scores) {
  int b, h, u;
  scores += blockIdx.z * g.scores_gs;
  pdl_wait();
  decode_unit(st, g.Hkv, blockIdx.x, b, h, u);
  if (g.pair && !(b & 1)) return;
  const int T = st.cu[b + 1] - st.cu[b];
  const int C = (T + g.c - 1) / g.c;
  const int nc = min(g.cpu, C - u * g.cpu);
  float* out = scores + ((int64_t)(b >> g.pair) * g.Hkv + h) * g.C_max + (int64_t)u * g.cpu;
  for (int ch = threadIdx.x; ch < nc; ch += blockDim.x) out[ch] = 0.f;
  pdl_trigger();
}

cudaError_t launch_finalize(const Plan& pl, const ScoreGeom& g, const SeqTable& st, float* rl,
                            const bin_t* bins, const float* lse, float* scores, int n_groups, cudaStream_t s) {
  (void)pl;
  if (g.n_units == 0 || n_groups == 0) return cudaSuccess;
  if (g.wG == 0)
    return launch_pdl(zero_scores_kernel, dim3(g.n_units, 1, n_groups), dim3(128), 0, s, g, st, scores);
  dim3 grid(g.n_units, (g.cpu + kFinChunks - 1) / kFinChunks, n_groups);
  if (lse != nullptr) {
    // a compile-time instance for w*G = 128 (LLaMA / Mistral-shaped groups with 32-query windows);
    // one for 448 measured slower than the run-time form
    if (g.wG == 128)
      return launch_pdl(finalize_kernel<true, 128>, grid, dim3(kFinThreads), 0, s, g, st, (const float*)rl, bins, lse,
                        scores);
    return launch_pdl(finalize_kernel<true, 0>, grid, dim3(kFinThreads), 0, s, g, st, (const float*)rl, bins, lse,
                      scores);
  }
  const size_t smem = (size_t)g.wG * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(finalize_kernel<false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(finalize_kernel<false, 0>, grid, dim3(kFinThreads), smem, s, g, st, (const float*)rl, bins, lse,
                    scores);
}

}  // namespace chunkkv
