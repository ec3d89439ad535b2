// C-ABI entry points of libchunkkv: argument checks, the workspace plan and the
// layer loop of ChunkKV §4.2 Algorithm 2 around §4.1 Algorithm 1.
#include <string.h>

#include <algorithm>

#include "common.cuh"

namespace chunkkv {

bool tc_supported(const Plan& pl);                                  // score_tc.cu
void tc_plan(Plan& pl);                                             // score_tc.cu
cudaError_t launch_score_tc(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* q,
                            const void* k, float* rl, float* bins, void* qpack, int32_t* err,
                            cudaStream_t s);

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;            // int32 device error word at offset 0

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

chunkkv_status check_params(const chunkkv_params* p) {
  if (p == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  if (p->B < 0 || p->Hq < 1 || p->Hkv < 1 || p->d < 1 || p->w < 0 || p->c < 1 || p->L_max < 0)
    return CHUNKKV_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return CHUNKKV_ERR_INVALID_ARG;
  if (p->dtype != CHUNKKV_F32 && p->dtype != CHUNKKV_BF16) return CHUNKKV_ERR_INVALID_ARG;
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
  pl.n_cap = n_cap;
  // scoring units: the tensor-core path sizes them for its tiles, the SIMT path
  // uses about 512 keys
  pl.use_tc = 0;
  pl.cpu = std::max(1, 512 / p->c);
  tc_plan(pl);                                    // may switch to the tensor-core geometry
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
  const size_t bins = align_up((size_t)pl.n_units * pl.cpu * pl.wG * sizeof(float));
  const size_t scores = align_up((size_t)p->B * p->Hkv * C_max * sizeof(float));
  const size_t qpack = pl.use_tc ? align_up((size_t)p->B * p->Hkv * pl.tc_mt * 128 * p->d * 2) : 0;
  pl.off_rl = 0;
  pl.off_bins = rl;
  pl.off_scores = rl + bins;
  pl.off_qpack = rl + bins + scores;
  pl.slot_bytes = rl + bins + scores + qpack;
  pl.header_bytes = kHeaderBytes;
  (void)n_layers;
  return CHUNKKV_OK;
}

ScoreGeom score_geom(const chunkkv_params* p, const Plan& pl) {
  ScoreGeom g;
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
  g.q_stride_b = p->q_stride_b;
  g.q_stride_w = p->q_stride_w;
  g.q_stride_h = p->q_stride_h;
  g.kv_stride_t = p->kv_stride_t;
  g.kv_stride_h = p->kv_stride_h;
  return g;
}

chunkkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CHUNKKV_OK : CHUNKKV_ERR_CUDA; }

// Scoring of one layer into `scores` through workspace slot `slot`.
cudaError_t run_score(const chunkkv_params* p, const Plan& pl, const SeqTable& st, const void* q,
                      const void* k, float* scores, char* ws, char* slot, cudaStream_t s) {
  const ScoreGeom g = score_geom(p, pl);
  float* rl = (float*)(slot + pl.off_rl);
  float* bins = (float*)(slot + pl.off_bins);
  cudaError_t e;
  if (pl.use_tc)
    e = launch_score_tc(pl, g, st, q, k, rl, bins, slot + pl.off_qpack, (int32_t*)ws, s);
  else
    e = launch_score_simt(pl, g, st, q, k, rl, bins, s);
  if (e != cudaSuccess) return e;
  return launch_finalize(pl, g, st, rl, bins, scores, s);
}

SelectGeom select_geom(const chunkkv_params* p, const Plan& pl) {
  SelectGeom sg;
  sg.Hkv = p->Hkv;
  sg.c = p->c;
  sg.w = p->w;
  sg.L_max = p->L_max;
  sg.C_max = pl.C_max;
  sg.n_cap = pl.n_cap;
  return sg;
}

GatherGeom gather_geom(const chunkkv_params* p, const Plan& pl) {
  GatherGeom gg;
  gg.Hkv = p->Hkv;
  gg.d = p->d;
  gg.elt = pl.elt;
  gg.n_cap = pl.n_cap;
  gg.kv_stride_t = p->kv_stride_t;
  gg.kv_stride_h = p->kv_stride_h;
  return gg;
}

cudaError_t run_gather(const chunkkv_params* p, const Plan& pl, const SeqTable& st, int n_layers,
                       const void* const* k, const void* const* v, void* const* ko, void* const* vo,
                       const int32_t* indices, const int32_t* counts, cudaStream_t s) {
  const GatherGeom gg = gather_geom(p, pl);
  const int nbh = pl.B * pl.Hkv;
  const int per_launch = std::max(1, std::min(CHUNKKV_MAX_GATHER_LAYERS, 65535 / std::max(1, nbh)));
  for (int l0 = 0; l0 < n_layers; l0 += per_launch) {
    GatherArgs ga;
    ga.n_layers = std::min(per_launch, n_layers - l0);
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
  *bytes = pl.header_bytes + pl.slot_bytes;
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
  if (ws_bytes < pl.header_bytes + pl.slot_bytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  char* w = (char*)ws;
  return cuda_status(run_score(p, pl, st, q_win, k, chunk_scores, w, w + pl.header_bytes,
                               (cudaStream_t)stream));
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
  return cuda_status(launch_select(pl, select_geom(p, pl), st, chunk_scores, indices, counts,
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
    if (!aligned16(k[l]) || !aligned16(v[l]) || !aligned16(k_out[l]) || !aligned16(v_out[l]) || !k[l] ||
        !v[l] || !k_out[l] || !v_out[l])
      return CHUNKKV_ERR_INVALID_ARG;
  return cuda_status(run_gather(p, pl, st, n_layers, k, v, k_out, v_out, indices, counts,
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
  if (ws_bytes < pl.header_bytes + pl.slot_bytes) return CHUNKKV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = (char*)ws;
  char* slot = w + pl.header_bytes;
  const size_t per_group_scores = (size_t)pl.B * pl.Hkv * pl.C_max;
  const size_t per_group_idx = (size_t)pl.B * pl.Hkv * pl.n_cap;
  const size_t per_group_cnt = (size_t)pl.B * pl.Hkv;
  const SelectGeom sg = select_geom(p, pl);
  for (int l0 = 0; l0 < n_layers; l0 += n_reuse) {
    const int grp = l0 / n_reuse;
    const int nl = std::min(n_reuse, n_layers - l0);
    float* sc = chunk_scores ? chunk_scores + grp * per_group_scores : (float*)(slot + pl.off_scores);
    int32_t* ix = indices ? indices + grp * per_group_idx : nullptr;
    int32_t* ct = counts + grp * per_group_cnt;
    cudaError_t e = run_score(p, pl, st, q_win[l0], k[l0], sc, w, slot, cs);
    if (e == cudaSuccess) e = launch_select(pl, sg, st, sc, ix, ct, cs);
    if (e == cudaSuccess)
      e = run_gather(p, pl, st, nl, k + l0, v + l0, k_out + l0, v_out + l0, ix, ct, cs);
    if (e != cudaSuccess) return CHUNKKV_ERR_CUDA;
  }
  return CHUNKKV_OK;
}

chunkkv_status chunkkv_status_check(void* ws, chunkkv_stream_t stream, int32_t* device_code) {
  if (ws == nullptr) return CHUNKKV_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return CHUNKKV_ERR_CUDA;
  int32_t code = 0;
  if (cudaMemcpy(&code, ws, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess) return CHUNKKV_ERR_CUDA;
  if (device_code) *device_code = code;
  if (code != 0) {
    if (cudaMemset(ws, 0, sizeof(int32_t)) != cudaSuccess) return CHUNKKV_ERR_CUDA;
    return CHUNKKV_ERR_TIMEOUT;
  }
  return CHUNKKV_OK;
}

}  // extern "C"
