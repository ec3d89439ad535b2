// Top-k chunk selection and kept-index construction.
//
// ChunkKV §4.1 Algorithm 1 steps 4-6: per (sequence b, KV head h) keep the
// k_b = min(L_max / c, C_b) chunks of largest score (ties to the lower chunk
// index), force in the last w tokens, and write the ascending, duplicate-free
// union of token positions.
//
// One CTA per (b, h):
//  1. radix select (4 passes of 8 bits) of the k-th largest order key, where
//     the order key is the fp32 bit pattern mapped to an unsigned integer that
//     sorts like the float (-0.0 canonicalised to +0.0);
//  2. one ordered sweep over the chunks: chunk i is kept if its key is above
//     the threshold, or equal to it and among the first `need_eq` equal keys in
//     index order (the tie rule);
//  3. expansion: with R = max(0, T - w) and s = floor(R / c), the kept chunks
//     below s are whole and land at rank * c; the chunk s straddling R (if kept)
//     contributes [s*c, R); the recent tokens [R, T) follow.  This order is
//     ascending by construction, so no sort is needed.
#include <cub/block/block_scan.cuh>

#include "fin.cuh"

namespace chunkkv {

constexpr int kSelThreads = 512;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) == 0u) u = 0u;                // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(SelectGeom sg, const __grid_constant__ SeqTable st, const float* __restrict__ scores,
              int32_t* __restrict__ indices, int32_t* __restrict__ counts) {
  using Scan = cub::BlockScan<int, kSelThreads>;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ int hist[256];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_remaining;
  __shared__ int sh_carry_eq, sh_carry_sel, sh_straddle;

  const int bh = blockIdx.x;
  const int b = bh / sg.Hkv;
  const int tid = threadIdx.x;
  const int T = st.cu[b + 1] - st.cu[b];
  const int c = sg.c;
  const int C = (T + c - 1) / c;
  const int k = min(sg.L_max / c, C);
  const float* A = scores + blockIdx.y * sg.scores_gs + (int64_t)bh * sg.C_max;
  int32_t* out = indices + blockIdx.y * sg.idx_gs + (int64_t)bh * sg.n_cap;
  counts += blockIdx.y * sg.cnt_gs;
  pdl_wait();

  // ---- 1. threshold key (k-th largest) and how many chunks equal to it are kept
  uint32_t thr = 0;
  int need_eq = 0;
  if (k > 0 && k < C) {
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < C; i += blockDim.x) {
        const uint32_t key = order_key(A[i]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      // descending digits: thread t holds the count of digit 255 - t
      const int cnt = tid < 256 ? hist[255 - tid] : 0;
      int incl;
      Scan(scan_tmp).InclusiveSum(cnt, incl);
      const int excl = incl - cnt;
      if (tid < 256 && excl < remaining && incl >= remaining) {
        sh_prefix = prefix | ((uint32_t)(255 - tid) << shift);
        sh_remaining = remaining - excl;
      }
      __syncthreads();
      prefix = sh_prefix;
      remaining = sh_remaining;
      mask |= 255u << shift;
      __syncthreads();
    }
    thr = prefix;
    need_eq = remaining;
  }

  // ---- 2./3. ordered sweep: keep flags, ranks, expansion of whole chunks below s
  const int Rs = max(0, T - sg.w);
  const int s = Rs / c;
  const int part = Rs - s * c;                      // tokens of chunk s below Rs
  if (tid == 0) { sh_carry_eq = 0; sh_carry_sel = 0; sh_straddle = 0; }
  __syncthreads();
  const int limit = min(C, s + 1);                  // chunks that can add tokens below Rs
  for (int base = 0; base < C && base < limit + 0; base += blockDim.x) {
    const int i = base + tid;
    int keep = 0, eq = 0;
    if (i < C && k > 0) {
      if (k >= C) {
        keep = 1;
      } else {
        const uint32_t key = order_key(A[i]);
        eq = key == thr;
        keep = key > thr;
      }
    }
    int eq_excl, eq_tot;
    Scan(scan_tmp).ExclusiveSum(eq, eq_excl, eq_tot);
    __syncthreads();
    if (eq && sh_carry_eq + eq_excl < need_eq) keep = 1;
    const int low = (i < s) ? keep : 0;             // whole chunks below Rs
    int rank_excl, low_tot;
    Scan(scan_tmp).ExclusiveSum(low, rank_excl, low_tot);
    if (low) {
      const int rank = sh_carry_sel + rank_excl;
      int32_t* o = out + (int64_t)rank * c;
      for (int t = 0; t < c; ++t) o[t] = i * c + t;
    }
    if (i == s && part > 0 && keep) sh_straddle = 1;
    __syncthreads();
    if (tid == 0) { sh_carry_eq += eq_tot; sh_carry_sel += low_tot; }
    __syncthreads();
  }
  const int n_low = sh_carry_sel;
  const int tail0 = n_low * c;
  const int strad = sh_straddle ? part : 0;
  for (int t = tid; t < strad; t += blockDim.x) out[tail0 + t] = s * c + t;
  const int rec0 = tail0 + strad;
  for (int t = tid; t < T - Rs; t += blockDim.x) out[rec0 + t] = Rs + t;
  if (tid == 0) counts[bh] = rec0 + (T - Rs);
  pdl_trigger();
}

// Register-resident variant for C <= 1024 * ITEMS: thread t holds the order keys
// of chunks t*ITEMS .. t*ITEMS+ITEMS-1 through the whole selection.  The
// threshold is found in three radix passes of 11, 11 and 10 bits over 2048-bin
// shared histograms: the first digit (exponent and leading mantissa bits) spreads
// similar-magnitude scores over many bins, so the shared atomics rarely collide,
// and the later passes only count the few keys that still match the prefix.  The
// ordered expansion needs two block scans.
constexpr int kSelBins = 2048;
constexpr int kSelRegThreads = 1024;

// Selection and index build of one (sequence, head) by the whole CTA (THREADS
// threads): thread t holds the order keys of chunks t*ITEMS .. t*ITEMS+ITEMS-1.
// A: the head's C chunk scores; out: its kept indices; count: its kept count.
template <int ITEMS, int THREADS = kSelRegThreads>
__device__ __forceinline__ void select_head(const SelectGeom& sg, int T, const float* A, int32_t* out,
                                            int32_t* count) {
  static_assert(kSelBins % THREADS == 0, "whole histogram bins per thread");
  using Scan = cub::BlockScan<int, THREADS>;
  constexpr int BPT = kSelBins / THREADS;                  // histogram bins per thread in the scan
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ int hist[kSelBins];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_remaining, sh_straddle;
  const int tid = threadIdx.x;
  const int c = sg.c;
  const int C = (T + c - 1) / c;
  const int k = min(sg.L_max / c, C);
  const int i0 = tid * ITEMS;

  uint32_t key[ITEMS];
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) key[j] = (i0 + j < C) ? order_key(__ldcg(A + i0 + j)) : 0u;

  // ---- threshold: the k-th largest key, and how many keys equal to it are kept
  uint32_t thr = 0;
  int need_eq = 0;
  if (k > 0 && k < C) {
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 1023u : 2047u;
      for (int i = tid; i < kSelBins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < ITEMS; ++j)
        if ((i0 + j < C) && ((key[j] & mask) == prefix)) atomicAdd(&hist[(key[j] >> shift) & dmask], 1);
      __syncthreads();
      // descending digits: thread t holds bins 2047 - BPT*t - i
      int cnt[BPT], tot = 0;
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        cnt[i] = hist[kSelBins - 1 - (BPT * tid + i)];
        tot += cnt[i];
      }
      int excl;
      Scan(scan_tmp).ExclusiveSum(tot, excl);
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        if (excl < remaining && excl + cnt[i] >= remaining) {
          sh_prefix = prefix | ((uint32_t)(kSelBins - 1 - (BPT * tid + i)) << shift);
          sh_remaining = remaining - excl;
        }
        excl += cnt[i];
      }
      __syncthreads();
      prefix = sh_prefix;
      remaining = sh_remaining;
      mask |= dmask << shift;
    }
    thr = prefix;
    need_eq = remaining;
  }

  // ---- keep flags: above the threshold, or equal to it and among the first need_eq in index order
  uint32_t keep = 0, eq = 0;
  int n_eq = 0;
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) {
    if (i0 + j < C && k > 0) {
      if (k >= C) {
        keep |= 1u << j;
      } else {
        if (key[j] > thr) keep |= 1u << j;
        if (key[j] == thr) { eq |= 1u << j; ++n_eq; }
      }
    }
  }
  if (tid == 0) sh_straddle = 0;
  int eq_base;
  Scan(scan_tmp).ExclusiveSum(n_eq, eq_base);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < ITEMS; ++j)
    if ((eq >> j) & 1u) {
      if (eq_base < need_eq) keep |= 1u << j;
      ++eq_base;
    }

  // ---- expansion: whole kept chunks below Rs = max(0, T - w) land at rank * c, in order
  const int Rs = max(0, T - sg.w);
  const int sc = Rs / c;
  const int part = Rs - sc * c;
  int n_low = 0;
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) n_low += ((keep >> j) & 1u) && (i0 + j < sc);
  int rank, low_tot;
  Scan(scan_tmp).ExclusiveSum(n_low, rank, low_tot);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) {
    const int i = i0 + j;
    if (((keep >> j) & 1u) && i < sc) {
      int32_t* o = out + (int64_t)rank * c;
      for (int t = 0; t < c; ++t) o[t] = i * c + t;
      ++rank;
    }
    if (i == sc && part > 0 && ((keep >> j) & 1u)) sh_straddle = 1;
  }
  __syncthreads();
  const int tail0 = low_tot * c;
  const int strad = sh_straddle ? part : 0;
  for (int t = tid; t < strad; t += blockDim.x) out[tail0 + t] = sc * c + t;
  const int rec0 = tail0 + strad;
  for (int t = tid; t < T - Rs; t += blockDim.x) out[rec0 + t] = Rs + t;
  if (tid == 0) *count = rec0 + (T - Rs);
}

// The same for kSelRegThreads * 16 < C <= kSelSmemChunks: the order keys sit in
// shared memory (dynamic, C words) instead of registers, thread t owning chunks
// t*n .. t*n+n-1 (n = ceil(C / 1024) <= 32), so the radix passes read them there
// and not from global memory as select_kernel does.
constexpr int kSelSmemChunks = 32 * kSelRegThreads;

__device__ __forceinline__ void select_head_smem(const SelectGeom& sg, int T, const float* A, int32_t* out,
                                                 int32_t* count, uint32_t* skey) {
  using Scan = cub::BlockScan<int, kSelRegThreads>;
  constexpr int BPT = kSelBins / kSelRegThreads;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ int hist[kSelBins];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_remaining, sh_straddle;
  const int tid = threadIdx.x;
  const int c = sg.c;
  const int C = (T + c - 1) / c;
  const int k = min(sg.L_max / c, C);
  const int n = (C + kSelRegThreads - 1) / kSelRegThreads;   // chunks per thread (<= 32)
  const int i0 = tid * n;
  for (int i = tid; i < C; i += kSelRegThreads) skey[i] = order_key(__ldcg(A + i));
  __syncthreads();

  // ---- threshold: the k-th largest key, and how many keys equal to it are kept
  uint32_t thr = 0;
  int need_eq = 0;
  if (k > 0 && k < C) {
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 1023u : 2047u;
      for (int i = tid; i < kSelBins; i += kSelRegThreads) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < C; i += kSelRegThreads) {
        const uint32_t key = skey[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1);
      }
      __syncthreads();
      // descending digits: thread t holds bins 2047 - BPT*t - i
      int cnt[BPT], tot = 0;
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        cnt[i] = hist[kSelBins - 1 - (BPT * tid + i)];
        tot += cnt[i];
      }
      int excl;
      Scan(scan_tmp).ExclusiveSum(tot, excl);
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        if (excl < remaining && excl + cnt[i] >= remaining) {
          sh_prefix = prefix | ((uint32_t)(kSelBins - 1 - (BPT * tid + i)) << shift);
          sh_remaining = remaining - excl;
        }
        excl += cnt[i];
      }
      __syncthreads();
      prefix = sh_prefix;
      remaining = sh_remaining;
      mask |= dmask << shift;
    }
    thr = prefix;
    need_eq = remaining;
  }

  // ---- keep flags of this thread's chunks (bit j: chunk i0 + j): above the threshold, or equal to
  // it and among the first need_eq in index order
  uint32_t keep = 0, eq = 0;
  int n_eq = 0;
  for (int j = 0; j < n; ++j) {
    const int i = i0 + j;
    if (i < C && k > 0) {
      if (k >= C) {
        keep |= 1u << j;
      } else {
        const uint32_t key = skey[i];
        if (key > thr) keep |= 1u << j;
        if (key == thr) { eq |= 1u << j; ++n_eq; }
      }
    }
  }
  if (tid == 0) sh_straddle = 0;
  int eq_base;
  Scan(scan_tmp).ExclusiveSum(n_eq, eq_base);
  __syncthreads();
  for (int j = 0; j < n; ++j)
    if ((eq >> j) & 1u) {
      if (eq_base < need_eq) keep |= 1u << j;
      ++eq_base;
    }

  // ---- expansion: whole kept chunks below Rs = max(0, T - w) land at rank * c, in order
  const int Rs = max(0, T - sg.w);
  const int sc = Rs / c;
  const int part = Rs - sc * c;
  int n_low = 0;
  for (int j = 0; j < n; ++j) n_low += ((keep >> j) & 1u) && (i0 + j < sc);
  int rank, low_tot;
  Scan(scan_tmp).ExclusiveSum(n_low, rank, low_tot);
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    const int i = i0 + j;
    if (((keep >> j) & 1u) && i < sc) {
      int32_t* o = out + (int64_t)rank * c;
      for (int t = 0; t < c; ++t) o[t] = i * c + t;
      ++rank;
    }
    if (i == sc && part > 0 && ((keep >> j) & 1u)) sh_straddle = 1;
  }
  __syncthreads();
  const int tail0 = low_tot * c;
  const int strad = sh_straddle ? part : 0;
  for (int t = tid; t < strad; t += kSelRegThreads) out[tail0 + t] = sc * c + t;
  const int rec0 = tail0 + strad;
  for (int t = tid; t < T - Rs; t += kSelRegThreads) out[rec0 + t] = Rs + t;
  if (tid == 0) *count = rec0 + (T - Rs);
}

__global__ void __launch_bounds__(kSelRegThreads)
select_smem_kernel(SelectGeom sg, const __grid_constant__ SeqTable st, const float* __restrict__ scores,
                   int32_t* __restrict__ indices, int32_t* __restrict__ counts) {
  extern __shared__ uint32_t skey[];
  const int bh = blockIdx.x;
  const int b = bh / sg.Hkv;
  const int T = st.cu[b + 1] - st.cu[b];
  const float* A = scores + blockIdx.y * sg.scores_gs + (int64_t)bh * sg.C_max;
  int32_t* out = indices + blockIdx.y * sg.idx_gs + (int64_t)bh * sg.n_cap;
  counts += blockIdx.y * sg.cnt_gs;
  pdl_wait();
  select_head_smem(sg, T, A, out, counts + bh, skey);
  pdl_trigger();
}

// THREADS < kSelRegThreads: several CTAs per SM, for calls with more heads than SMs.
template <int ITEMS, int THREADS>
__global__ void __launch_bounds__(THREADS, kSelRegThreads / THREADS)
select_reg_kernel(SelectGeom sg, const __grid_constant__ SeqTable st, const float* __restrict__ scores,
                  int32_t* __restrict__ indices, int32_t* __restrict__ counts) {
  const int bh = blockIdx.x;
  const int b = bh / sg.Hkv;
  const int T = st.cu[b + 1] - st.cu[b];
  const float* A = scores + blockIdx.y * sg.scores_gs + (int64_t)bh * sg.C_max;
  int32_t* out = indices + blockIdx.y * sg.idx_gs + (int64_t)bh * sg.n_cap;
  counts += blockIdx.y * sg.cnt_gs;
  pdl_wait();
  select_head<ITEMS, THREADS>(sg, T, A, out, counts + bh);
  pdl_trigger();
}

// Log-sum-exp, finalisation and selection of one (sequence, head, reuse group)
// in one CTA, for calls with enough heads to fill the GPU with such CTAs: the
// row log-sum-exps go to shared memory, the chunk scores to the score array
// (read back from L2 by the selection in the same CTA), and no other launch sits
// between the scoring kernel and the gather.  Shared memory: lse[wG], then the
// partial (M, S) pairs of the P = kSelRegThreads / wG thread groups that split
// the units of every row when wG < kSelRegThreads.
template <int ITEMS>
__global__ void __launch_bounds__(kSelRegThreads)
head_kernel(ScoreGeom g, SelectGeom sg, const __grid_constant__ SeqTable st, const float* __restrict__ rl,
            const bin_t* __restrict__ bins, float* __restrict__ scores, int32_t* __restrict__ indices,
            int32_t* __restrict__ counts) {
  extern __shared__ float hsh[];
  const int bh = blockIdx.x;
  const int b = bh / g.Hkv, h = bh - b * g.Hkv;
  rl += blockIdx.y * g.rl_gs;
  bins += blockIdx.y * g.bins_gs;
  float* A = scores + blockIdx.y * g.scores_gs + (int64_t)bh * g.C_max;
  int32_t* out = indices + blockIdx.y * sg.idx_gs + (int64_t)bh * sg.n_cap;
  counts += blockIdx.y * sg.cnt_gs;
  const int T = st.cu[b + 1] - st.cu[b];
  const int C = (T + g.c - 1) / g.c;
  const int U = st.uoff[b + 1] - st.uoff[b];
  pdl_wait();

  // 1. base-2 log-sum-exp of every window row of the head over its U units
  float* lse_s = hsh;
  float* part = hsh + g.wG;
  const int P = g.wG < kSelRegThreads ? kSelRegThreads / g.wG : 1;
  const int64_t ustride = (int64_t)g.Hkv * 2 * g.wG;            // between units of one head
  const float* rl_head = rl + ((int64_t)st.uoff[b] * g.Hkv + h) * 2 * g.wG;
  for (int t = threadIdx.x; t < g.wG * P; t += kSelRegThreads) {
    const int r = t % g.wG, p = t / g.wG;
    const float* base = rl_head + r;
    float M = -INFINITY, S = 0.f;
    int v = p;
    for (; v + 3 * P < U; v += 4 * P) {
      float Rv[4], lv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        Rv[i] = base[(v + i * P) * ustride];
        lv[i] = base[(v + i * P) * ustride + g.wG];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) lse_merge(M, S, Rv[i], lv[i]);
    }
    for (; v < U; v += P) lse_merge(M, S, base[v * ustride], base[v * ustride + g.wG]);
    if (P == 1) {
      lse_s[r] = M + log2f(S);
    } else {
      part[2 * t] = M;
      part[2 * t + 1] = S;
    }
  }
  if (P > 1) {
    __syncthreads();
    for (int r = threadIdx.x; r < g.wG; r += kSelRegThreads) {
      float M = -INFINITY, S = 0.f;
      for (int p = 0; p < P; ++p) lse_merge(M, S, part[2 * (p * g.wG + r)], part[2 * (p * g.wG + r) + 1]);
      lse_s[r] = M + log2f(S);
    }
  }
  __syncthreads();

  // 2. chunk scores of every unit, kFinGroup chunks per warp step
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // (eight-chunk steps even for small w*G: a head's units are short, and with one CTA per head the
  // sixteen-chunk steps leave more of each unit's last step empty; measured slower at T = 32768)
  const int spu = (g.cpu + kFinGroup - 1) / kFinGroup;            // warp steps per unit
  for (int it = warp; it < U * spu; it += kSelRegThreads / 32) {
    const int u = it / spu;
    const int ch0 = (it - u * spu) * kFinGroup;
    const int m = min(kFinGroup, min(g.cpu, C - u * g.cpu) - ch0);
    if (m <= 0) continue;                                          // past the end of the last unit
    const int gu = (st.uoff[b] + u) * g.Hkv + h;
    fin_group<true>(bins + ((int64_t)gu * g.cpu + ch0) * g.wG, g.wG, m, nullptr, rl + (int64_t)gu * 2 * g.wG,
                    lse_s, A + (int64_t)u * g.cpu + ch0, lane);
  }
  __syncthreads();                                                // the scores are visible to the whole CTA

  // 3. selection and index build
  select_head<ITEMS>(sg, T, A, out, counts + bh);
  pdl_trigger();
}

cudaError_t launch_select(const Plan& pl, const SelectGeom& sg, const SeqTable& st, const float* scores,
                          int32_t* indices, int32_t* counts, int n_groups, cudaStream_t s) {
  const int n = pl.B * pl.Hkv;
  if (n == 0 || n_groups == 0) return cudaSuccess;
  const dim3 grid(n, n_groups);
  // Each CTA's selection is a chain of block-wide steps; with more heads than SMs, smaller CTAs
  // (several per SM) overlap the chains of different heads.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return cudaErrorInvalidDevice;
  if ((int64_t)n * n_groups > sms) {
    if (pl.C_max <= 256 * 8)
      return launch_pdl(select_reg_kernel<8, 256>, grid, dim3(256), 0, s, sg, st, scores, indices, counts);
    if (pl.C_max <= 512 * 8)
      return launch_pdl(select_reg_kernel<8, 512>, grid, dim3(512), 0, s, sg, st, scores, indices, counts);
    if (pl.C_max <= 512 * 12)
      return launch_pdl(select_reg_kernel<12, 512>, grid, dim3(512), 0, s, sg, st, scores, indices, counts);
  }
  if (pl.C_max <= kSelRegThreads * 4)
    return launch_pdl(select_reg_kernel<4, kSelRegThreads>, grid, dim3(kSelRegThreads), 0, s, sg, st, scores, indices,
                      counts);
  if (pl.C_max <= kSelRegThreads * 13)            // 13 keys a thread spill less than 16 (128K: 13108 chunks)
    return launch_pdl(select_reg_kernel<13, kSelRegThreads>, grid, dim3(kSelRegThreads), 0, s, sg, st, scores,
                      indices, counts);
  if (pl.C_max <= kSelRegThreads * 16)
    return launch_pdl(select_reg_kernel<16, kSelRegThreads>, grid, dim3(kSelRegThreads), 0, s, sg, st, scores,
                      indices, counts);
  if (pl.C_max <= kSelSmemChunks) {
    const size_t smem = (size_t)pl.C_max * sizeof(uint32_t);
    const cudaError_t e =
        cudaFuncSetAttribute(select_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_smem_kernel, grid, dim3(kSelRegThreads), smem, s, sg, st, scores, indices, counts);
  }
  return launch_pdl(select_kernel, grid, dim3(kSelThreads), 0, s, sg, st, scores, indices, counts);
}

// Whether head_kernel can take the log-sum-exp, finalisation and selection of a
// call: window rows and a register-resident selection fit one 1024-thread CTA,
// and the call's (group, sequence, head) CTAs make one wave that fills at least
// three quarters of the GPU's SMs (one CTA per SM).  With more heads than SMs
// the separate kernels are faster: a head's CTA spends a fixed time on its
// log-sum-exp and selection, wave after wave.
bool head_path(const Plan& pl, int n_groups, int sms) {
  if (pl.wG <= 0 || pl.C_max > kSelRegThreads * 16 || sms <= 0) return false;
  const int64_t heads = (int64_t)pl.B * pl.Hkv * n_groups;
  return heads <= sms && 4 * heads >= 3 * (int64_t)sms;
}

cudaError_t launch_head(const Plan& pl, const ScoreGeom& g, const SelectGeom& sg, const SeqTable& st,
                        const float* rl, const bin_t* bins, float* scores, int32_t* indices, int32_t* counts,
                        int n_groups, cudaStream_t s) {
  const int P = pl.wG < kSelRegThreads ? kSelRegThreads / pl.wG : 1;
  const size_t smem = (size_t)pl.wG * (P > 1 ? 1 + 2 * P : 1) * sizeof(float);   // at most 16 KB (wG <= 4096)
  const dim3 grid(pl.B * pl.Hkv, n_groups);
  if (pl.C_max <= kSelRegThreads * 4)
    return launch_pdl(head_kernel<4>, grid, dim3(kSelRegThreads), smem, s, g, sg, st, rl, bins, scores, indices,
                      counts);
  return launch_pdl(head_kernel<16>, grid, dim3(kSelRegThreads), smem, s, g, sg, st, rl, bins, scores, indices,
                    counts);
}

}  // namespace chunkkv
