// chunkkv_score_noalloc: window scoring for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they score: code that
// runs inside a memory pool or arena that owns every device byte, allocator
// hooks and custom memory managers (calling back into the allocator would
// recurse or deadlock), or embedded runtimes whose memory budget is fixed at
// start-up.  They also cannot hand us a workspace if they have none to spare.
// This entry point runs the portable SIMT scoring kernel and the per-unit
// finalisation with their scratch (per-unit reference exponents, row sums and
// per-chunk bins) in one file-scope device array of kNoAllocScratchBytes, so a
// call needs nothing beyond its inputs and its output.
//
// Costs and rules of that array:
//  * it is part of the library's device image: every GPU that loads the
//    library holds kNoAllocScratchBytes of device memory until the process exits;
//  * all calls share it, and it keeps whatever the last call left there; a call
//    reads only values that the same call wrote first, so nothing in it has to
//    start at zero;
//  * two calls whose kernels can overlap on the GPU (different streams, or
//    different host threads) race on it and corrupt each other's scores;
//  * on each device, the first call looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture begins.
#include <mutex>

#include "common.cuh"

namespace chunkkv {
namespace {

// the size the header states (CHUNKKV_NOALLOC_SCRATCH_BYTES), so that the limit
// this file enforces is the documented one
constexpr size_t kNoAllocScratchBytes = CHUNKKV_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes == (size_t(16) << 20), "16 MiB of static scratch");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_setup_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_setup_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_setup_ptr[dev] = ptr;
  }
  *out = g_setup_ptr[dev];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace chunkkv

using namespace chunkkv;

extern "C" chunkkv_status chunkkv_score_noalloc(const chunkkv_params* p, const void* q_win, const void* k,
                                                float* chunk_scores, chunkkv_stream_t stream) {
  size_t ws_bytes = 0;
  chunkkv_status s = chunkkv_workspace_size(p, 1, 1, &ws_bytes);     // validates every parameter
  if (s != CHUNKKV_OK) return s;
  const int G = p->Hq / p->Hkv;
  const int wG = p->w * G;
  const int cpu = p->c >= 512 ? 1 : 512 / p->c;                       // SIMT unit: ~512 keys
  static thread_local SeqTable st;
  st.B = p->B;
  int64_t units = 0;
  int C_max = 0;
  for (int b = 0; b <= p->B; ++b) {
    st.cu[b] = p->cu_seqlens ? p->cu_seqlens[b] : 0;
    st.uoff[b] = (int32_t)units;
    if (b < p->B) {
      const int T = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
      const int C = (int)(((int64_t)T + p->c - 1) / p->c);
      C_max = C > C_max ? C : C_max;
      units += (C + cpu - 1) / cpu;
    }
  }
  const int64_t n_units = units * p->Hkv;
  if (n_units == 0) return CHUNKKV_OK;
  const size_t rl_bytes = align256((size_t)n_units * 2 * wG * sizeof(float));
  const size_t bin_bytes = align256((size_t)n_units * cpu * wG * sizeof(bin_t));
  if (rl_bytes + bin_bytes > kNoAllocScratchBytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  if ((wG > 0 && (!q_win || ((uintptr_t)q_win & 15u))) || !k || ((uintptr_t)k & 15u) || !chunk_scores)
    return CHUNKKV_ERR_INVALID_ARG;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return CHUNKKV_ERR_CUDA;

  Plan pl = {};
  pl.B = p->B;
  pl.Hkv = p->Hkv;
  pl.elt = p->dtype == CHUNKKV_BF16 ? 2 : 4;
  ScoreGeom g = {};
  g.Hq = p->Hq;
  g.Hkv = p->Hkv;
  g.G = G;
  g.d = p->d;
  g.w = p->w;
  g.wG = wG;
  g.c = p->c;
  g.cpu = cpu;
  g.ku = cpu * p->c;
  g.n_units = (int32_t)n_units;
  g.C_max = C_max;
  g.alpha = (float)(1.4426950408889634 / sqrt((double)p->d));
  g.causal = p->causal_window;
  g.q_stride_b = p->q_stride_b;
  g.q_stride_w = p->q_stride_w;
  g.q_stride_h = p->q_stride_h;
  g.kv_stride_t = p->kv_stride_t;
  g.kv_stride_h = p->kv_stride_h;
  g.rl_gs = g.bins_gs = g.lse_gs = g.scores_gs = 0;      // a single group
  float* rl = (float*)base;
  bin_t* bins = (bin_t*)((char*)base + rl_bytes);
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = launch_score_simt(pl, g, st, q_win, k, rl, bins, cs);
  if (e == cudaSuccess) e = launch_finalize(pl, g, st, rl, bins, nullptr, chunk_scores, 1, cs);
  return e == cudaSuccess ? CHUNKKV_OK : CHUNKKV_ERR_CUDA;
}
