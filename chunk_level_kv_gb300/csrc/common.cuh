// Shared definitions of the ChunkKV CUDA library: launch geometry, the sequence
// table that travels as a kernel argument, and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <climits>

#include "chunkkv.h"

namespace chunkkv {

// Limits of this build (checked on the host before any launch).
constexpr int kMaxWG = 4096;          // window rows per KV head, w * G
constexpr int kMaxD = 256;            // head dimension

// Chunk bins are stored as 16-bit unsigned floats: the upper 16 bits, rounded
// half up at the 11th significant bit (a relative error of at most 2^-11), of the
// fp32 pattern of the bin's value scaled by 2^-kBinShift.  A bin is a sum of
// 2^(t - R) >= 0 over one chunk; the scoring kernels form the scaled values
// directly, as 2^(t - R') with the shifted reference R' = R + kBinShift, which
// is the reference they also write out.  A bin b in [2^-40, 2^23) of R is then
// a normal float in [2^-126, 2^-63), whose exponent field (1 .. 63) and top ten
// mantissa bits are the code; smaller bins become fp32 subnormals or zero (an
// absolute error of at most 2^-51 of R), and code 0 is zero.  Bins from
// (1 - 2^-12) 2^23 up would round past 16 bits: the tensor-core kernel keeps the
// bins it keeps below (1 - 2^-10) 2^23 of R (it rescales a row before its sum
// passes that), the portable kernel saturates (its bins stay below the chunk
// length).
using bin_t = uint16_t;
constexpr int kBinShift = 86;
// Two integer ops: for scaled bins below 2^-63 (the tensor-core kernel's).
__device__ __forceinline__ bin_t bin_encode(float v) { return (bin_t)((__float_as_uint(v) + 0x1000u) >> 13); }
// Saturating at the largest code, for bins without a bound.
__device__ __forceinline__ bin_t bin_encode_sat(float v) {
  return (bin_t)min((__float_as_uint(v) + 0x1000u) >> 13, 0xFFFFu);
}
// The scaled value of a code.
__device__ __forceinline__ float bin_decode(uint32_t code) { return __uint_as_float(code << 13); }
// The two bins packed in a 32-bit word (low half first), two integer ops a bin.
__device__ __forceinline__ float2 bin_decode2(uint32_t v) {
  return make_float2(__uint_as_float((v << 13) & 0x1FFFE000u), __uint_as_float((v >> 3) & 0x1FFFE000u));
}

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
  int32_t causal;     // window query q sees keys 0 .. T - w + q only (chunkkv_params.causal_window)
  // 1: the sequences come in pairs (2i = the kept prefix of cache i, 2i + 1 = its new tail) for an
  // incremental pass during decoding: both read the window rows of cache i, the row log-sum-exp
  // spans both, and only the tail has chunk scores (at index i)
  int32_t pair;
  int64_t q_stride_b, q_stride_w, q_stride_h;
  int64_t kv_stride_t, kv_stride_h;
  // Distance (in floats) between the buffers of consecutive reuse groups, for the
  // kernels that handle every group of a call in one launch (blockIdx.z = group).
  int64_t rl_gs, bins_gs, lse_gs, scores_gs;     // group strides: floats, bin_t, floats, floats
};

// Selection / index-build geometry (blockIdx.y = reuse group).
struct SelectGeom {
  int32_t Hkv, c, w, L_max, C_max, n_cap;
  int64_t scores_gs, idx_gs, cnt_gs;            // per-group strides in elements
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
  int32_t n_reuse, l0;                          // layer l0 + i of a launch uses group (l0 + i) / n_reuse
  int32_t pair;                                 // paired sequences (see ScoreGeom): only tails, lists at i
  int64_t kv_stride_t, kv_stride_h;
  int64_t idx_gs, cnt_gs;                       // per-group strides of indices / counts
};

// Device error codes written to the first word of the workspace.
enum DeviceError : int32_t {
  kDevOk = 0,
  kDevTimeoutTmaProducer = 0x101,
  kDevTimeoutMma = 0x102,
  kDevTimeoutEpilogue = 0x103,
  kDevTimeoutSelftest = 0x1FF,      // chunkkv_selftest_wait_timeout
  kDevMisalignedSmem = 0x201,
};

// The workspace header (256 bytes, zero-filled before the workspace's first use):
// int32 word 0 is the device error word; words kSchedWord and kSchedWord + 1 are
// the tensor-core scoring launch's item counter and count of finished CTAs, which
// the launch's last CTA sets back to zero.
constexpr int kSchedWord = 4;

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

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation: it calls pdl_wait() before it touches
// memory that the previous kernel in the stream writes or reads, and
// pdl_trigger() once its own work is done, so the next kernel's launch and
// prologue overlap this kernel's drain but never take resources this kernel
// still needs.  Both are no-ops when a kernel is launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// ----------------------------------------------------------------- host side

// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger).
// Kernels launched through launch_pdl by this process (chunkkv_launch_count).
extern std::atomic<unsigned long long> g_launch_count;

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// Workspace plan shared by the C-ABI entry points and the launchers.
struct Plan {
  int32_t B, Hkv, G, d, w, wG, c, L_max, elt;
  int32_t C_max, n_cap, max_T;
  int32_t cpu, ku, n_units;
  int32_t use_tc;                 // tensor-core scoring kernel
  int32_t tc_mt;                  // 128-row M tiles of the window rows (tensor-core path)
  int32_t tc_base_chunks;         // chunks in the smallest whole-tile unit (tensor-core path)
  int32_t tc_tile_n;              // keys per tile of the tensor-core kernel
  int32_t n_groups;               // reuse groups of the call (scoring layers)
  size_t slot_bytes;              // one group's scratch: rl, bins, lse
  size_t off_rl, off_bins, off_lse;                 // inside a slot
  size_t off_slots, off_qpack, off_scores;          // regions of the workspace (after the header)
  size_t scores_group_bytes;                        // one group's chunk scores (scores region holds all)
  size_t qpack_group_bytes;                         // one layer's packed window rows (tensor-core path)
  size_t header_bytes;
  size_t total_bytes;
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_score_simt(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* q,
                              const void* k, float* rl, bin_t* bins, cudaStream_t s);
cudaError_t launch_finalize(const Plan& pl, const ScoreGeom& g, const SeqTable& st, float* rl,
                            const bin_t* bins, const float* lse, float* scores, int n_groups, cudaStream_t s);
cudaError_t launch_lse(const ScoreGeom& g, const SeqTable& st, const float* rl, float* lse, int n_groups,
                       cudaStream_t s);
cudaError_t launch_select(const Plan& pl, const SelectGeom& sg, const SeqTable& st, const float* scores,
                          int32_t* indices, int32_t* counts, int n_groups, cudaStream_t s);
cudaError_t launch_gather(const Plan& pl, const GatherGeom& gg, const SeqTable& st, const GatherArgs& ga,
                          const int32_t* indices, const int32_t* counts, cudaStream_t s);

}  // namespace chunkkv
