// Shared definitions of the ChunkKV CUDA library: launch geometry, the sequence
// table that travels as a kernel argument, and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/chunkkv.h"

namespace chunkkv {

// Limits of this build (checked on the host before any launch).
constexpr int kMaxWG = 4096;          // window rows per KV head, w * G
constexpr int kMaxD = 256;            // head dimension

// Per-sequence table passed by value: token offsets and scoring-unit offsets.
// A scoring unit is one (sequence b, KV head h, run of `cpu` chunks); units of
// one sequence are numbered u = 0 .. U_b-1 and all heads of a unit are
// adjacent: global unit id gu = (uoff[b] + u) * Hkv + h.
struct SeqTable {
  int32_t B;
  int32_t cu[CHUNKKV_MAX_BATCH + 1];
  int32_t uoff[CHUNKKV_MAX_BATCH + 1];
};

// Geometry of one scoring layer.
struct ScoreGeom {
  int32_t Hq, Hkv, G, d, w, wG, c;
  int32_t cpu;        // chunks per unit
  int32_t ku;         // keys per unit = cpu * c
  int32_t n_units;    // Hkv * uoff[B]
  int32_t C_max;      // chunk capacity of the score array
  float alpha;        // log2(e) / sqrt(d): logits are handled as base-2 exponents
  int64_t q_stride_b, q_stride_w, q_stride_h;
  int64_t kv_stride_t, kv_stride_h;
};

// Selection / index-build geometry.
struct SelectGeom {
  int32_t Hkv, c, w, L_max, C_max, n_cap;
};

// Layers moved by one gather launch.
struct GatherArgs {
  int32_t n_layers;
  const void* k[CHUNKKV_MAX_GATHER_LAYERS];
  const void* v[CHUNKKV_MAX_GATHER_LAYERS];
  void* ko[CHUNKKV_MAX_GATHER_LAYERS];
  void* vo[CHUNKKV_MAX_GATHER_LAYERS];
};

struct GatherGeom {
  int32_t Hkv, d, elt, n_cap;
  int64_t kv_stride_t, kv_stride_h;
};

// Device error codes written to the first word of the workspace.
enum DeviceError : int32_t {
  kDevOk = 0,
  kDevTimeoutTmaProducer = 0x101,
  kDevTimeoutMma = 0x102,
  kDevTimeoutEpilogue = 0x103,
};

// Decode a global unit id into (b, h, u).
__device__ __forceinline__ void decode_unit(const SeqTable& st, int Hkv, int gu, int& b, int& h, int& u) {
  h = gu % Hkv;
  int ul = gu / Hkv;
  int lo = 0, hi = st.B;          // find b with uoff[b] <= ul < uoff[b+1]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (st.uoff[mid] <= ul) lo = mid; else hi = mid;
  }
  b = lo;
  u = ul - st.uoff[b];
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// ----------------------------------------------------------------- host side

// Workspace plan shared by the C-ABI entry points and the launchers.
struct Plan {
  int32_t B, Hkv, G, d, w, wG, c, L_max, elt;
  int32_t C_max, n_cap;
  int32_t cpu, ku, n_units;
  int32_t use_tc;                 // tensor-core scoring kernel
  int32_t tc_mt;                  // 128-row M tiles of the window rows (tensor-core path)
  size_t slot_bytes;              // one scoring slot
  size_t off_rl, off_bins, off_scores, off_qpack;   // inside a slot
  size_t header_bytes;
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_score_simt(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* q,
                              const void* k, float* rl, float* bins, cudaStream_t s);
cudaError_t launch_finalize(const Plan& pl, const ScoreGeom& g, const SeqTable& st, float* rl,
                            const float* bins, float* scores, cudaStream_t s);
cudaError_t launch_select(const Plan& pl, const SelectGeom& sg, const SeqTable& st, const float* scores,
                          int32_t* indices, int32_t* counts, cudaStream_t s);
cudaError_t launch_gather(const Plan& pl, const GatherGeom& gg, const SeqTable& st, const GatherArgs& ga,
                          const int32_t* indices, const int32_t* counts, cudaStream_t s);

}  // namespace chunkkv
