// C-ABI entry points of libchunkkv: argument checks, the workspace plan and the
// layer loop of ChunkKV §4.2 Algorithm 2 around §4.1 Algorithm 1.
#include <string.h>

#include <algorithm>
#include <vector>

#include "common.cuh"

namespace chunkkv {

std::atomic<unsigned long long> g_launch_count{0};

void tc_plan(Plan& pl);                                             // score_tc.cu
cudaError_t launch_wait_selftest(int32_t* err, long long timeout, cudaStream_t s);   // score_tc.cu
cudaError_t launch_overlap(const SeqTable& st, int Hkv, int n_cap, int n_lists, int max_T, const int32_t* indices,
                           const int32_t* counts, int32_t* inter, int32_t* uni, cudaStream_t s);   // overlap.cu
cudaError_t launch_pack_q(const Plan& pl, const ScoreGeom& g, const void* const* q_layers, int n_layers,
                          void* qpack, cudaStream_t s);
cudaError_t launch_score_tc(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* const* q_groups,
                            const void* const* k_groups, int n_groups, int64_t slot_bytes, float* rl, bin_t* bins,
                            const void* qpack, int32_t* err, cudaStream_t s, int mode, const float* lse);
cudaError_t launch_sum_partials(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const float* part,
                                int64_t slot_bytes, float* scores, int n_groups, cudaStream_t s);   // score_tc.cu
bool tc_q_direct(const Plan& pl, const ScoreGeom& g, const void* q);                   // score_tc.cu
bool head_path(const Plan& pl, int n_groups, int sms);                                 // select.cu
cudaError_t launch_head(const Plan& pl, const ScoreGeom& g, const SelectGeom& sg, const SeqTable& st,
                        const float* rl, const bin_t* bins, float* scores, int32_t* indices, int32_t* counts,
                        int n_groups, cudaStream_t s);

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;            // int32 device error word at offset 0
constexpr int kItemTiles = 2;                   // fixed cost of a scoring work item, in key tiles

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

// The tensor-core scoring kernel reads a scoring layer's keys through a TMA
// tensor map, which needs device memory; everything else the kernels read or
// write with plain loads and stores, which may also be host memory that the
// GPU addresses directly (pinned or registered).
bool device_memory(const void* ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

// SMs of the current device.  Without a visible device (sizes computed on a
// host that has no GPU) a GB300's 152 is assumed; a plan made for another SM
// count then asks for a different workspace size, which the size check catches.
int current_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

chunkkv_status check_params(const chunkkv_params* p) {
  if (p == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  if (p->B < 0 || p->Hq < 1 || p->Hkv < 1 || p->d < 1 || p->w < 0 || p->c < 1 || p->L_max < 0)
    return CHUNKKV_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return CHUNKKV_ERR_INVALID_ARG;
  if (p->dtype != CHUNKKV_F32 && p->dtype != CHUNKKV_BF16) return CHUNKKV_ERR_INVALID_ARG;
  if (p->causal_window != 0 && p->causal_window != 1) return CHUNKKV_ERR_INVALID_ARG;
  if (p->B > CHUNKKV_MAX_BATCH || p->d > kMaxD) return CHUNKKV_ERR_UNSUPPORTED;
  if ((int64_t)p->w * (p->Hq / p->Hkv) > kMaxWG) return CHUNKKV_ERR_UNSUPPORTED;
  if ((int64_t)p->B * p->Hkv > 65535) return CHUNKKV_ERR_UNSUPPORTED;
  const int elt = p->dtype == CHUNKKV_BF16 ? 2 : 4;
  if ((p->d * elt) % 16 != 0) return CHUNKKV_ERR_INVALID_ARG;
  const int64_t strides[5] = {p->q_stride_b, p->q_stride_w, p->q_stride_h, p->kv_stride_t, p->kv_stride_h};
  for (int64_t s : strides)
    if (s < 0 || (s * elt) % 16 != 0) return CHUNKKV_ERR_INVALID_ARG;
  if (p->B > 0) {
    if (p->cu_seqlens == nullptr || p->cu_seqlens[0] != 0) return CHUNKKV_ERR_INVALID_ARG;
    for (int b = 0; b < p->B; ++b)
      if (p->cu_seqlens[b + 1] < p->cu_seqlens[b]) return CHUNKKV_ERR_INVALID_ARG;
  }
  return CHUNKKV_OK;
}

chunkkv_status make_plan(const chunkkv_params* p, int n_layers, int n_reuse, Plan& pl, SeqTable* st) {
  chunkkv_status s = check_params(p);
  if (s != CHUNKKV_OK) return s;
  if (n_layers < 0 || n_reuse < 1) return CHUNKKV_ERR_INVALID_ARG;
  memset(&pl, 0, sizeof(pl));
  pl.B = p->B;
  pl.Hkv = p->Hkv;
  pl.G = p->Hq / p->Hkv;
  pl.d = p->d;
  pl.w = p->w;
  pl.wG = p->w * pl.G;
  pl.c = p->c;
  pl.L_max = p->L_max;
  pl.elt = p->dtype == CHUNKKV_BF16 ? 2 : 4;
  int max_T = 0, C_max = 0, n_cap = 0;
  for (int b = 0; b < p->B; ++b) {
    const int T = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
    const int C = (int)(((int64_t)T + p->c - 1) / p->c);
    const int k = std::min(p->L_max / p->c, C);
    const int64_t cap = std::min<int64_t>(T, (int64_t)k * p->c + std::min(p->w, T));
    max_T = std::max(max_T, T);
    C_max = std::max(C_max, C);
    n_cap = std::max<int>(n_cap, (int)cap);
  }
  pl.C_max = C_max;
  pl.max_T = max_T;
  pl.n_cap = n_cap;
  // scoring units: the tensor-core path sizes them for its tiles, the SIMT path
  // uses about 512 keys
  pl.use_tc = 0;
  pl.cpu = std::max(1, 512 / p->c);
  tc_plan(pl);                                    // may switch to the tensor-core geometry
  if (pl.use_tc) {
    // Unit length for the persistent tensor-core grid: the multiple m of the
    // base unit that minimises (waves of work items) x (tiles per item + the
    // fixed cost of an item, kItemTiles tiles: reference maximum, window-row
    // reload, pipeline refill) with two CTAs per SM (304 slots on a GB300); ties
    // go to longer units.
    const int slots = 2 * current_sm_count();
    const int64_t per_unit_items = (int64_t)p->Hkv * pl.tc_mt;
    const int base_tiles = pl.tc_base_chunks * p->c / pl.tc_tile_n;
    int64_t best_cost = INT64_MAX;
    for (int m = 1; m <= 64; ++m) {
      const int cpu = pl.tc_base_chunks * m;
      int64_t items = 0;
      for (int b = 0; b < p->B; ++b) {
        const int T = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
        const int64_t C = ((int64_t)T + p->c - 1) / p->c;
        items += (C + cpu - 1) / cpu * per_unit_items;
      }
      if (items == 0) break;
      const int64_t cost = (items + slots - 1) / slots * ((int64_t)m * base_tiles + kItemTiles);
      if (cost <= best_cost) {
        best_cost = cost;
        pl.cpu = cpu;
      }
      if (items <= per_unit_items) break;          // one unit per sequence already
    }
  }
  pl.ku = pl.cpu * p->c;
  int64_t units = 0;
  if (st) st->B = p->B;
  for (int b = 0; b <= p->B; ++b) {
    if (st) {
      st->cu[b] = p->cu_seqlens ? p->cu_seqlens[b] : 0;
      st->uoff[b] = (int32_t)units;
    }
    if (b < p->B) {
      const int T = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
      const int C = (int)(((int64_t)T + p->c - 1) / p->c);
      units += (C + pl.cpu - 1) / pl.cpu;
    }
  }
  if (units * p->Hkv > INT32_MAX / 2) return CHUNKKV_ERR_UNSUPPORTED;
  pl.n_units = (int32_t)(units * p->Hkv);
  const size_t rl = align_up((size_t)pl.n_units * 2 * pl.wG * sizeof(float));
  const size_t bins = align_up((size_t)pl.n_units * pl.cpu * pl.wG * sizeof(bin_t));
  const size_t lse = align_up((size_t)p->B * p->Hkv * pl.wG * sizeof(float));
  pl.n_groups = n_layers > 0 ? (n_layers + n_reuse - 1) / n_reuse : 1;
  // Workspace: [header | one scratch slot per reuse group | packed window rows
  // per group (tensor-core path) | chunk scores per group].  Every group has its
  // own slot, so the scoring of all groups can run back to back before the
  // (batched) log-sum-exp, finalisation, selection and gather.
  pl.off_rl = 0;
  pl.off_bins = rl;
  pl.off_lse = rl + bins;
  pl.slot_bytes = rl + bins + lse;
  pl.qpack_group_bytes = pl.use_tc ? align_up((size_t)p->B * p->Hkv * pl.tc_mt * 128 * p->d * 2) : 0;
  pl.scores_group_bytes = align_up((size_t)p->B * p->Hkv * C_max * sizeof(float));
  pl.header_bytes = kHeaderBytes;
  pl.off_slots = 0;
  pl.off_qpack = pl.slot_bytes * pl.n_groups;
  pl.off_scores = pl.off_qpack + pl.qpack_group_bytes * pl.n_groups;
  pl.total_bytes = pl.header_bytes + pl.off_scores + pl.scores_group_bytes * pl.n_groups;
  return CHUNKKV_OK;
}

ScoreGeom score_geom(const chunkkv_params* p, const Plan& pl) {
  ScoreGeom g = {};
  g.Hq = p->Hq;
  g.Hkv = p->Hkv;
  g.G = pl.G;
  g.d = p->d;
  g.w = p->w;
  g.wG = pl.wG;
  g.c = p->c;
  g.cpu = pl.cpu;
  g.ku = pl.ku;
  g.n_units = pl.n_units;
  g.C_max = pl.C_max;
  g.alpha = (float)(1.4426950408889634 / sqrt((double)p->d));
  g.causal = p->causal_window;
  g.q_stride_b = p->q_stride_b;
  g.q_stride_w = p->q_stride_w;
  g.q_stride_h = p->q_stride_h;
  g.kv_stride_t = p->kv_stride_t;
  g.kv_stride_h = p->kv_stride_h;
  g.rl_gs = g.lse_gs = (int64_t)(pl.slot_bytes / sizeof(float));
  g.bins_gs = (int64_t)(pl.slot_bytes / sizeof(bin_t));
  g.scores_gs = (int64_t)(pl.scores_group_bytes / sizeof(float));
  return g;
}

chunkkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CHUNKKV_OK : CHUNKKV_ERR_CUDA; }

// Token-level chunks (c = 1) on the tensor-core path take two passes over the
// keys instead of one: the first forms each row's (R, l) pairs only, the
// log-sum-exp kernel their lse, and the second sums every key's probabilities
// over the window rows directly.  A bin per logit (16 bits per row and key,
// written and read back) would cost more than reading the keys twice.  Not with
// the causal window or paired sequences (they keep the single pass).  The second
// pass's partial arrays (fp32 per token and KV head, one per warp of window rows:
// 4 ceil(wG / 32) bytes per token and head) go where the bins would be (2 wG
// bytes per token and head, the units covering every token): they fit for wG >= 2.
bool two_pass(const Plan& pl, const ScoreGeom& g) {
  return pl.use_tc && pl.c == 1 && !g.causal && !g.pair && pl.wG >= 2;
}

// Scoring of n_groups reuse groups into consecutive scratch slots from `slots`.
// q and k hold each group's scoring layer; on the tensor-core path one
// persistent launch covers all groups, reading the window rows from q itself
// (qpack null) or from their packed copy in qpack.
cudaError_t run_score_groups(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* const* q,
                             const void* const* k, int n_groups, char* slots, const void* qpack, int32_t* err,
                             cudaStream_t s) {
  float* rl = (float*)(slots + pl.off_rl);
  bin_t* bins = (bin_t*)(slots + pl.off_bins);
  const int64_t slot_gs = (int64_t)(pl.slot_bytes / sizeof(float));
  if (pl.use_tc)
    return launch_score_tc(pl, g, st, q, k, n_groups, (int64_t)pl.slot_bytes, rl, bins, qpack, err, s,
                           two_pass(pl, g) ? 1 : 0, nullptr);
  for (int i = 0; i < n_groups; ++i) {
    cudaError_t e = launch_score_simt(pl, g, st, q[i], k[i], rl + i * slot_gs,
                                      (bin_t*)((char*)bins + i * pl.slot_bytes), s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Phase events of chunkkv_set_phase_events (this host thread), recorded only
// inside chunkkv_compress_layers.
thread_local void* t_phase_ev[CHUNKKV_PHASE_EVENTS];
thread_local int t_phase_n = 0;
thread_local bool t_in_compress = false;

cudaError_t phase_mark(int i, cudaStream_t s) {
  if (!t_in_compress || t_phase_n == 0) return cudaSuccess;
  return cudaEventRecord((cudaEvent_t)t_phase_ev[i], s);
}

// Log-sum-exp and finalisation of n_groups consecutive slots into their chunk
// scores; for two-pass token-level chunks the finalisation is the second pass
// over the keys (q, k, qpack, err as for run_score_groups) and the sum of its
// partial arrays.
cudaError_t run_post_score(const Plan& pl, const ScoreGeom& g, const SeqTable& st, char* slots, float* scores,
                           int n_groups, cudaStream_t s, const void* const* q, const void* const* k,
                           const void* qpack, int32_t* err) {
  float* rl = (float*)(slots + pl.off_rl);
  float* lse = (float*)(slots + pl.off_lse);
  bin_t* bins = (bin_t*)(slots + pl.off_bins);
  cudaError_t e = launch_lse(g, st, rl, lse, n_groups, s);
  if (e == cudaSuccess) e = phase_mark(3, s);
  if (e != cudaSuccess) return e;
  if (two_pass(pl, g)) {
    e = launch_score_tc(pl, g, st, q, k, n_groups, (int64_t)pl.slot_bytes, rl, bins, qpack, err, s, 2, lse);
    if (e != cudaSuccess) return e;
    return launch_sum_partials(pl, g, st, (const float*)bins, (int64_t)pl.slot_bytes, scores, n_groups, s);
  }
  return launch_finalize(pl, g, st, rl, bins, lse, scores, n_groups, s);
}

SelectGeom select_geom(const chunkkv_params* p, const Plan& pl) {
  SelectGeom sg = {};
  sg.Hkv = p->Hkv;
  sg.c = p->c;
  sg.w = p->w;
  sg.L_max = p->L_max;
  sg.C_max = pl.C_max;
  sg.n_cap = pl.n_cap;
  sg.scores_gs = (int64_t)pl.B * pl.Hkv * pl.C_max;
  sg.idx_gs = (int64_t)pl.B * pl.Hkv * pl.n_cap;
  sg.cnt_gs = (int64_t)pl.B * pl.Hkv;
  return sg;
}

GatherGeom gather_geom(const chunkkv_params* p, const Plan& pl) {
  GatherGeom gg = {};
  gg.Hkv = p->Hkv;
  gg.d = p->d;
  gg.elt = pl.elt;
  gg.n_cap = pl.n_cap;
  gg.kv_stride_t = p->kv_stride_t;
  gg.kv_stride_h = p->kv_stride_h;
  gg.n_reuse = 1;
  gg.l0 = 0;
  gg.idx_gs = (int64_t)pl.B * pl.Hkv * pl.n_cap;
  gg.cnt_gs = (int64_t)pl.B * pl.Hkv;
  return gg;
}

// Gather of n_layers layers; layer l uses index group l / n_reuse.
cudaError_t run_gather(const chunkkv_params* p, const Plan& pl, const SeqTable& st, int n_layers, int n_reuse,
                       const void* const* k, const void* const* v, void* const* ko, void* const* vo,
                       const int32_t* indices, const int32_t* counts, cudaStream_t s) {
  GatherGeom gg = gather_geom(p, pl);
  gg.n_reuse = n_reuse;
  const int nbh = pl.B * pl.Hkv;
  const int per_launch = std::max(1, std::min(CHUNKKV_MAX_GATHER_LAYERS, 65535 / std::max(1, nbh)));
  for (int l0 = 0; l0 < n_layers; l0 += per_launch) {
    GatherArgs ga;
    ga.n_layers = std::min(per_launch, n_layers - l0);
    gg.l0 = l0;
    for (int i = 0; i < ga.n_layers; ++i) {
      ga.k[i] = k[l0 + i];
      ga.v[i] = v[l0 + i];
      ga.ko[i] = ko[l0 + i];
      ga.vo[i] = vo[l0 + i];
    }
    cudaError_t e = launch_gather(pl, gg, st, ga, indices, counts, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace chunkkv

using namespace chunkkv;

extern "C" {

const char* chunkkv_status_string(chunkkv_status s) {
  switch (s) {
    case CHUNKKV_OK: return "ok";
    case CHUNKKV_ERR_INVALID_ARG: return "invalid argument";
    case CHUNKKV_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case CHUNKKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CHUNKKV_ERR_CUDA: return "CUDA error";
    case CHUNKKV_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

chunkkv_status chunkkv_out_capacity(const chunkkv_params* p, int32_t* n_cap_max, int32_t* C_max) {
  Plan pl;
  chunkkv_status s = make_plan(p, 1, 1, pl, nullptr);
  if (s != CHUNKKV_OK) return s;
  if (n_cap_max) *n_cap_max = pl.n_cap;
  if (C_max) *C_max = pl.C_max;
  return CHUNKKV_OK;
}

chunkkv_status chunkkv_workspace_size(const chunkkv_params* p, int32_t n_layers, int32_t n_reuse,
                                      size_t* bytes) {
  if (bytes == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  Plan pl;
  chunkkv_status s = make_plan(p, n_layers, n_reuse, pl, nullptr);
  if (s != CHUNKKV_OK) return s;
  *bytes = pl.total_bytes;
  return CHUNKKV_OK;
}

int32_t chunkkv_score_path(const chunkkv_params* p) {
  Plan pl;
  if (make_plan(p, 1, 1, pl, nullptr) != CHUNKKV_OK) return -1;
  return pl.use_tc;
}

chunkkv_status chunkkv_score(const chunkkv_params* p, const void* q_win, const void* k,
                             float* chunk_scores, void* ws, size_t ws_bytes, chunkkv_stream_t stream) {
  Plan pl;
  static thread_local SeqTable st;
  chunkkv_status s = make_plan(p, 1, 1, pl, &st);
  if (s != CHUNKKV_OK) return s;
  if (pl.n_units == 0) return CHUNKKV_OK;
  if ((pl.wG > 0 && (!q_win || !aligned16(q_win))) || !k || !chunk_scores || !ws || !aligned16(k) ||
      !aligned16(ws))
    return CHUNKKV_ERR_INVALID_ARG;
  if (ws_bytes < pl.total_bytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  if (pl.use_tc && !device_memory(k)) return CHUNKKV_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = (char*)ws;
  char* base = w + pl.header_bytes;
  char* slot = base + pl.off_slots;
  char* qpack = base + pl.off_qpack;
  ScoreGeom g = score_geom(p, pl);
  cudaError_t e = cudaSuccess;
  // window rows straight from q_win when a tensor map can address them (w divides 128 and q_win is
  // device memory), else packed first with plain loads (q_win may be host memory the GPU addresses)
  const bool direct = tc_q_direct(pl, g, q_win) && device_memory(q_win);
  if (pl.use_tc && pl.wG > 0 && !direct) {
    const void* ql[1] = {q_win};
    e = launch_pack_q(pl, g, ql, 1, qpack, cs);
  }
  if (e == cudaSuccess)
    e = run_score_groups(pl, g, st, &q_win, &k, 1, slot, direct ? nullptr : qpack, (int32_t*)w, cs);
  if (e == cudaSuccess)
    e = run_post_score(pl, g, st, slot, chunk_scores, 1, cs, &q_win, &k, direct ? nullptr : qpack, (int32_t*)w);
  return cuda_status(e);
}

chunkkv_status chunkkv_select(const chunkkv_params* p, const float* chunk_scores, int32_t* indices,
                              int32_t* counts, chunkkv_stream_t stream) {
  Plan pl;
  static thread_local SeqTable st;
  chunkkv_status s = make_plan(p, 1, 1, pl, &st);
  if (s != CHUNKKV_OK) return s;
  if (pl.B * pl.Hkv == 0) return CHUNKKV_OK;
  if (!counts || (pl.C_max > 0 && !chunk_scores) || (pl.n_cap > 0 && !indices))
    return CHUNKKV_ERR_INVALID_ARG;
  return cuda_status(launch_select(pl, select_geom(p, pl), st, chunk_scores, indices, counts, 1,
                                   (cudaStream_t)stream));
}

chunkkv_status chunkkv_gather(const chunkkv_params* p, int32_t n_layers, const int32_t* indices,
                              const int32_t* counts, const void* const* k, const void* const* v,
                              void* const* k_out, void* const* v_out, chunkkv_stream_t stream) {
  Plan pl;
  static thread_local SeqTable st;
  chunkkv_status s = make_plan(p, 1, 1, pl, &st);
  if (s != CHUNKKV_OK) return s;
  if (n_layers < 1 || n_layers > CHUNKKV_MAX_GATHER_LAYERS) return CHUNKKV_ERR_INVALID_ARG;
  if (pl.B * pl.Hkv == 0 || pl.n_cap == 0) return CHUNKKV_OK;
  if (!indices || !counts || !k || !v || !k_out || !v_out) return CHUNKKV_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!k[l] || !v[l] || !k_out[l] || !v_out[l] || !aligned16(k[l]) || !aligned16(v[l]) ||
        !aligned16(k_out[l]) || !aligned16(v_out[l]))
      return CHUNKKV_ERR_INVALID_ARG;
  // every layer of this call shares the one index list: group (l / n_layers) = 0
  return cuda_status(run_gather(p, pl, st, n_layers, n_layers, k, v, k_out, v_out, indices, counts,
                                (cudaStream_t)stream));
}

chunkkv_status chunkkv_compress_layers(const chunkkv_params* p, int32_t n_layers, int32_t n_reuse,
                                       const void* const* q_win, const void* const* k,
                                       const void* const* v, void* const* k_out, void* const* v_out,
                                       int32_t* indices, int32_t* counts, float* chunk_scores,
                                       void* ws, size_t ws_bytes, chunkkv_stream_t stream) {
  Plan pl;
  static thread_local SeqTable st;
  chunkkv_status s = make_plan(p, n_layers, n_reuse, pl, &st);
  if (s != CHUNKKV_OK) return s;
  if (n_layers < 1) return CHUNKKV_ERR_INVALID_ARG;
  if (pl.B * pl.Hkv == 0) return CHUNKKV_OK;
  if (!q_win || !k || !v || !k_out || !v_out || !counts || !ws || !aligned16(ws))
    return CHUNKKV_ERR_INVALID_ARG;
  if (pl.n_cap > 0 && !indices) return CHUNKKV_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    if (l % n_reuse == 0 && pl.wG > 0 && (!q_win[l] || !aligned16(q_win[l])))
      return CHUNKKV_ERR_INVALID_ARG;
    if (!k[l] || !v[l] || !k_out[l] || !v_out[l] || !aligned16(k[l]) || !aligned16(v[l]) ||
        !aligned16(k_out[l]) || !aligned16(v_out[l]))
      return CHUNKKV_ERR_INVALID_ARG;
  }
  if (ws_bytes < pl.total_bytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  if (pl.use_tc)
    for (int l = 0; l < n_layers; l += n_reuse)
      if (!device_memory(k[l])) return CHUNKKV_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = (char*)ws;
  char* base = w + pl.header_bytes;
  const int n_groups = pl.n_groups;
  ScoreGeom g = score_geom(p, pl);
  float* scores = chunk_scores ? chunk_scores : (float*)(base + pl.off_scores);
  if (chunk_scores) g.scores_gs = (int64_t)pl.B * pl.Hkv * pl.C_max;
  // One stream, every launch chained by programmatic dependent launch:
  //  1. the window rows of every scoring layer packed in one launch (tensor-core path, only
  //     when the scoring kernel cannot read them from q_win itself);
  //  2. the scoring kernel of each reuse group, back to back, each into its own slot;
  //  3. log-sum-exp and finalisation of all groups in one launch each;
  //  4. top-k selection and index build of every (group, sequence, head) in one launch;
  //     (3 and 4 are one launch, head_kernel, when the call has enough heads to fill the GPU)
  //  5. the gather of every layer (layer l with index group l / n_reuse).
  cudaError_t e = cudaSuccess;
  struct InCompress {                   // phase events are recorded only inside this call
    InCompress() { t_in_compress = true; }
    ~InCompress() { t_in_compress = false; }
  } in_compress;
  static thread_local std::vector<const void*> qsel, ksel;
  qsel.resize(n_groups);
  ksel.resize(n_groups);
  for (int i = 0; i < n_groups; ++i) {
    qsel[i] = q_win[i * n_reuse];
    ksel[i] = k[i * n_reuse];
  }
  // window rows straight from q_win when a tensor map can address them (w divides 128, every scoring
  // layer's q_win in device memory), else packed first with plain loads; every layer has the same
  // strides and was checked for 16-byte alignment, so the first decides the map's shape
  bool direct = tc_q_direct(pl, g, qsel[0]);
  for (int i = 0; direct && i < n_groups; ++i) direct = device_memory(qsel[i]);
  const void* qpack = direct ? nullptr : base + pl.off_qpack;
  e = phase_mark(0, cs);
  if (e == cudaSuccess && pl.use_tc && pl.wG > 0 && !direct) e = launch_pack_q(pl, g, qsel.data(), n_groups, base + pl.off_qpack, cs);
  if (e == cudaSuccess) e = phase_mark(1, cs);
  if (e == cudaSuccess)
    e = run_score_groups(pl, g, st, qsel.data(), ksel.data(), n_groups, base + pl.off_slots, qpack, (int32_t*)w, cs);
  if (e == cudaSuccess) e = phase_mark(2, cs);
  SelectGeom sg = select_geom(p, pl);
  sg.scores_gs = g.scores_gs;
  if (!two_pass(pl, g) && head_path(pl, n_groups, current_sm_count())) {
    // enough (group, sequence, head) CTAs to fill the GPU: log-sum-exp, finalisation and selection
    // of a head in one CTA (the lse and select phases are then empty)
    if (e == cudaSuccess) e = phase_mark(3, cs);
    if (e == cudaSuccess) {
      char* slots = base + pl.off_slots;
      e = launch_head(pl, g, sg, st, (const float*)(slots + pl.off_rl), (const bin_t*)(slots + pl.off_bins), scores,
                      indices, counts, n_groups, cs);
    }
    if (e == cudaSuccess) e = phase_mark(4, cs);
  } else {
    if (e == cudaSuccess)
      e = run_post_score(pl, g, st, base + pl.off_slots, scores, n_groups, cs, qsel.data(), ksel.data(), qpack,
                         (int32_t*)w);
    if (e == cudaSuccess) e = phase_mark(4, cs);
    if (e == cudaSuccess) e = launch_select(pl, sg, st, scores, indices, counts, n_groups, cs);
  }
  if (e == cudaSuccess) e = phase_mark(5, cs);
  if (e == cudaSuccess) e = run_gather(p, pl, st, n_layers, n_reuse, k, v, k_out, v_out, indices, counts, cs);
  if (e == cudaSuccess) e = phase_mark(6, cs);
  return cuda_status(e);
}

// ----------------------------------------------------------------- incremental pass during decoding
namespace chunkkv {
namespace {

// The two tables of an incremental pass (reading R12): `pv` describes 2B sequences, 2b the kept
// prefix of cache b and 2b + 1 its new tail, on which the scoring, the log-sum-exp and the
// finalisation run (keys of the prefix count in each row's normaliser only); `pt` describes the B
// tails alone, which the selection and the output layout use.
struct TailTables {
  chunkkv_params pv, pt;
  int32_t cu_v[2 * CHUNKKV_MAX_BATCH + 1];
  int32_t cu_t[CHUNKKV_MAX_BATCH + 1];
};

chunkkv_status tail_tables(const chunkkv_params* p, const int32_t* n_prev, TailTables& t) {
  chunkkv_status s = check_params(p);
  if (s != CHUNKKV_OK) return s;
  if (p->causal_window) return CHUNKKV_ERR_UNSUPPORTED;
  if (p->B > 0 && n_prev == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  if (2 * p->B > CHUNKKV_MAX_BATCH || (int64_t)2 * p->B * p->Hkv > 65535) return CHUNKKV_ERR_UNSUPPORTED;
  t.cu_t[0] = 0;
  for (int b = 0; b < p->B; ++b) {
    const int T = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
    if (n_prev[b] < 0 || n_prev[b] > T) return CHUNKKV_ERR_INVALID_ARG;
    t.cu_v[2 * b] = p->cu_seqlens[b];
    t.cu_v[2 * b + 1] = p->cu_seqlens[b] + n_prev[b];
    t.cu_t[b + 1] = t.cu_t[b] + (T - n_prev[b]);
  }
  t.cu_v[2 * p->B] = p->B > 0 ? p->cu_seqlens[p->B] : 0;
  t.pv = *p;
  t.pv.B = 2 * p->B;
  t.pv.cu_seqlens = t.cu_v;
  t.pt = *p;
  t.pt.cu_seqlens = t.cu_t;
  return CHUNKKV_OK;
}

}  // namespace
}  // namespace chunkkv

chunkkv_status chunkkv_tail_sizes(const chunkkv_params* p, const int32_t* n_prev, int32_t n_layers, int32_t n_reuse,
                                  int32_t* n_cap_max, int32_t* C_max, size_t* ws_bytes) {
  static thread_local TailTables t;
  chunkkv_status s = tail_tables(p, n_prev, t);
  if (s != CHUNKKV_OK) return s;
  if (n_layers < 1 || n_reuse < 1) return CHUNKKV_ERR_INVALID_ARG;
  Plan pv, pt;
  if ((s = make_plan(&t.pv, n_layers, n_reuse, pv, nullptr)) != CHUNKKV_OK) return s;
  if ((s = make_plan(&t.pt, 1, 1, pt, nullptr)) != CHUNKKV_OK) return s;
  if (n_cap_max) *n_cap_max = pt.n_cap;
  if (C_max) *C_max = pt.C_max;
  if (ws_bytes) *ws_bytes = pv.total_bytes;
  return CHUNKKV_OK;
}

chunkkv_status chunkkv_compress_tail(const chunkkv_params* p, const int32_t* n_prev, int32_t n_layers, int32_t n_reuse,
                                     const void* const* q_win, const void* const* k, const void* const* v,
                                     void* const* k_out, void* const* v_out, int32_t* indices, int32_t* counts,
                                     float* chunk_scores, void* ws, size_t ws_bytes, chunkkv_stream_t stream) {
  static thread_local TailTables t;
  static thread_local SeqTable st_v, st_t;
  chunkkv_status s = tail_tables(p, n_prev, t);
  if (s != CHUNKKV_OK) return s;
  if (n_layers < 1 || n_reuse < 1) return CHUNKKV_ERR_INVALID_ARG;
  Plan pv, pt;
  if ((s = make_plan(&t.pv, n_layers, n_reuse, pv, &st_v)) != CHUNKKV_OK) return s;
  if ((s = make_plan(&t.pt, 1, 1, pt, &st_t)) != CHUNKKV_OK) return s;
  if (pt.B * pt.Hkv == 0) return CHUNKKV_OK;
  if (!q_win || !k || !v || !k_out || !v_out || !counts || !ws || !aligned16(ws)) return CHUNKKV_ERR_INVALID_ARG;
  if (pt.n_cap > 0 && !indices) return CHUNKKV_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    if (l % n_reuse == 0 && pv.wG > 0 && (!q_win[l] || !aligned16(q_win[l]))) return CHUNKKV_ERR_INVALID_ARG;
    if (!k[l] || !v[l] || !k_out[l] || !v_out[l] || !aligned16(k[l]) || !aligned16(v[l]) || !aligned16(k_out[l]) ||
        !aligned16(v_out[l]))
      return CHUNKKV_ERR_INVALID_ARG;
  }
  if (ws_bytes < pv.total_bytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  if (pv.use_tc)
    for (int l = 0; l < n_layers; l += n_reuse)
      if (!device_memory(k[l])) return CHUNKKV_ERR_INVALID_ARG;
  const int n_groups = pv.n_groups;
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = (char*)ws;
  char* base = w + pv.header_bytes;
  char* slots = base + pv.off_slots;
  ScoreGeom g = score_geom(&t.pv, pv);
  g.pair = 1;
  g.C_max = pt.C_max;                       // chunk scores of the tails only, [groups, B, Hkv, C_max]
  g.scores_gs = (int64_t)pt.B * pt.Hkv * pt.C_max;
  float* scores = chunk_scores ? chunk_scores : (float*)(base + pv.off_scores);
  static thread_local std::vector<const void*> qsel, ksel;
  qsel.resize(n_groups);
  ksel.resize(n_groups);
  for (int i = 0; i < n_groups; ++i) {
    qsel[i] = q_win[i * n_reuse];
    ksel[i] = k[i * n_reuse];
  }
  cudaError_t e = cudaSuccess;
  struct InCompress {                   // phase events are recorded inside this call too
    InCompress() { t_in_compress = true; }
    ~InCompress() { t_in_compress = false; }
  } in_compress;
  bool direct = tc_q_direct(pv, g, qsel[0]);
  for (int i = 0; direct && i < n_groups; ++i) direct = device_memory(qsel[i]);
  char* qpack = direct ? nullptr : base + pv.off_qpack;
  e = phase_mark(0, cs);
  if (e == cudaSuccess && pv.use_tc && pv.wG > 0 && !direct) e = launch_pack_q(pv, g, qsel.data(), n_groups, qpack, cs);
  if (e == cudaSuccess) e = phase_mark(1, cs);
  if (e == cudaSuccess) e = run_score_groups(pv, g, st_v, qsel.data(), ksel.data(), n_groups, slots, qpack, (int32_t*)w, cs);
  if (e == cudaSuccess) e = phase_mark(2, cs);
  if (e == cudaSuccess)
    e = run_post_score(pv, g, st_v, slots, scores, n_groups, cs, qsel.data(), ksel.data(), qpack, (int32_t*)w);
  if (e == cudaSuccess) e = phase_mark(4, cs);
  SelectGeom sg = select_geom(&t.pt, pt);
  if (e == cudaSuccess) e = launch_select(pt, sg, st_t, scores, indices, counts, n_groups, cs);
  if (e == cudaSuccess) e = phase_mark(5, cs);
  if (e == cudaSuccess && pt.n_cap > 0) {
    // every layer of every (cache, head) of the paired table, layer l with group l / n_reuse;
    // the kept prefixes append nothing
    GatherGeom gg = gather_geom(&t.pt, pt);
    gg.pair = 1;
    gg.n_reuse = n_reuse;
    Plan pg = pt;
    pg.B = pv.B;
    const int per_launch = std::max(1, std::min(CHUNKKV_MAX_GATHER_LAYERS, 65535 / std::max(1, pv.B * pv.Hkv)));
    for (int l0 = 0; l0 < n_layers && e == cudaSuccess; l0 += per_launch) {
      GatherArgs ga;
      ga.n_layers = std::min(per_launch, n_layers - l0);
      gg.l0 = l0;
      for (int i = 0; i < ga.n_layers; ++i) {
        ga.k[i] = k[l0 + i];
        ga.v[i] = v[l0 + i];
        ga.ko[i] = k_out[l0 + i];
        ga.vo[i] = v_out[l0 + i];
      }
      e = launch_gather(pg, gg, st_v, ga, indices, counts, cs);
    }
  }
  if (e == cudaSuccess) e = phase_mark(6, cs);
  return cuda_status(e);
}

chunkkv_status chunkkv_set_phase_events(void* const* events, int32_t n_events) {
  if (n_events == 0) {
    t_phase_n = 0;
    return CHUNKKV_OK;
  }
  if (n_events != CHUNKKV_PHASE_EVENTS || events == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  for (int i = 0; i < CHUNKKV_PHASE_EVENTS; ++i)
    if (events[i] == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  for (int i = 0; i < CHUNKKV_PHASE_EVENTS; ++i) t_phase_ev[i] = events[i];
  t_phase_n = CHUNKKV_PHASE_EVENTS;
  return CHUNKKV_OK;
}

chunkkv_status chunkkv_layer_overlap(const chunkkv_params* p, int32_t n_lists, const int32_t* indices,
                                     const int32_t* counts, int32_t* inter, int32_t* uni, chunkkv_stream_t stream) {
  Plan pl;
  static thread_local SeqTable st;
  chunkkv_status s = make_plan(p, 1, 1, pl, &st);
  if (s != CHUNKKV_OK) return s;
  if (n_lists < 1) return CHUNKKV_ERR_INVALID_ARG;
  if (n_lists == 1 || pl.B * pl.Hkv == 0) return CHUNKKV_OK;
  if (!counts || !inter || !uni || (pl.n_cap > 0 && !indices)) return CHUNKKV_ERR_INVALID_ARG;
  if ((size_t)(pl.max_T + 31) / 32 * sizeof(uint32_t) > 227 * 1024) return CHUNKKV_ERR_UNSUPPORTED;
  if ((int64_t)n_lists - 1 > 65535) return CHUNKKV_ERR_UNSUPPORTED;
  return cuda_status(launch_overlap(st, pl.Hkv, pl.n_cap, n_lists, pl.max_T, indices, counts, inter, uni,
                                    (cudaStream_t)stream));
}

chunkkv_status chunkkv_selftest_wait_timeout(void* ws, size_t ws_bytes, chunkkv_stream_t stream) {
  if (ws == nullptr || !aligned16(ws) || ws_bytes < kHeaderBytes) return CHUNKKV_ERR_INVALID_ARG;
  // about a millisecond of clock64 cycles, instead of the scoring kernel's two seconds
  return cuda_status(launch_wait_selftest((int32_t*)ws, 2000000LL, (cudaStream_t)stream));
}

uint64_t chunkkv_launch_count(void) { return chunkkv::g_launch_count.load(std::memory_order_relaxed); }

chunkkv_status chunkkv_status_check(void* ws, chunkkv_stream_t stream, int32_t* device_code) {
  if (ws == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  // everything on the caller's stream, so that no other stream is waited for
  int32_t code = 0;
  if (cudaMemcpyAsync(&code, ws, sizeof(code), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return CHUNKKV_ERR_CUDA;
  if (device_code) *device_code = code;
  if (code != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), cs) != cudaSuccess || cudaStreamSynchronize(cs) != cudaSuccess)
      return CHUNKKV_ERR_CUDA;
    return CHUNKKV_ERR_TIMEOUT;
  }
  return CHUNKKV_OK;
}

}  // extern "C"
