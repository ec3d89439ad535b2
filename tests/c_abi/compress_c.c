/*
 * A caller of libchunkkv.so written in plain C (C99, no Python, no torch): it
 * reads one small batch from files, allocates its device buffers itself with
 * the CUDA runtime, runs chunkkv_compress_layers (ChunkKV §4.2 Algorithm 2
 * around §4.1 Algorithm 1) through the C-ABI of include/chunkkv.h, checks the
 * device status word and writes every output back to files.
 *
 * usage: compress_c DIR
 *   DIR/meta.txt   "B Hq Hkv d w c L_max n_layers n_reuse dtype" then B+1 cu_seqlens
 *   DIR/q<l>.bin   window queries of layer l [B, w, Hq, d] (raw elements; bf16 = 2 bytes)
 *   DIR/k<l>.bin, DIR/v<l>.bin   keys and values [T_total, Hkv, d]
 * writes DIR/out_meta.txt "n_cap C_max", DIR/counts.bin, DIR/indices.bin,
 * DIR/scores.bin (groups x B x Hkv x C_max fp32) and DIR/ko<l>.bin, DIR/vo<l>.bin.
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "chunkkv.h"

#define CHECK_CUDA(x)                                                             \
  do {                                                                            \
    cudaError_t e_ = (x);                                                         \
    if (e_ != cudaSuccess) {                                                      \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                    \
      return 2;                                                                   \
    }                                                                             \
  } while (0)
#define CHECK_CKV(x)                                                              \
  do {                                                                            \
    chunkkv_status s_ = (x);                                                      \
    if (s_ != CHUNKKV_OK) {                                                       \
      fprintf(stderr, "%s: %s\n", #x, chunkkv_status_string(s_));                 \
      return 3;                                                                   \
    }                                                                             \
  } while (0)

static void* read_file(const char* dir, const char* name, size_t* n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  *n = (size_t)ftell(f);
  fseek(f, 0, SEEK_SET);
  void* p = malloc(*n ? *n : 1);
  if (p && fread(p, 1, *n, f) != *n) {
    free(p);
    p = NULL;
  }
  fclose(f);
  return p;
}

static int write_file(const char* dir, const char* name, const void* p, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 0;
  const int ok = fwrite(p, 1, n, f) == n;
  fclose(f);
  return ok;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s DIR\n", argv[0]);
    return 1;
  }
  const char* dir = argv[1];
  char path[4096];
  snprintf(path, sizeof path, "%s/meta.txt", dir);
  FILE* mf = fopen(path, "r");
  if (!mf) {
    fprintf(stderr, "cannot read %s\n", path);
    return 1;
  }
  int B, Hq, Hkv, d, w, c, L_max, n_layers, n_reuse, dtype;
  if (fscanf(mf, "%d %d %d %d %d %d %d %d %d %d", &B, &Hq, &Hkv, &d, &w, &c, &L_max, &n_layers, &n_reuse,
             &dtype) != 10 || B < 1 || B > 64 || n_layers < 1 || n_layers > 64 || n_reuse < 1) {
    fprintf(stderr, "bad meta.txt\n");
    return 1;
  }
  int32_t cu[65];
  for (int b = 0; b <= B; ++b)
    if (fscanf(mf, "%d", &cu[b]) != 1) {
      fprintf(stderr, "bad cu_seqlens\n");
      return 1;
    }
  fclose(mf);
  const size_t elt = dtype == CHUNKKV_BF16 ? 2 : 4;

  chunkkv_params p;
  memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.d = d;
  p.w = w;
  p.c = c;
  p.L_max = L_max;
  p.dtype = dtype;
  p.cu_seqlens = cu;
  p.q_stride_b = (int64_t)w * Hq * d;
  p.q_stride_w = (int64_t)Hq * d;
  p.q_stride_h = d;
  p.kv_stride_t = (int64_t)Hkv * d;
  p.kv_stride_h = d;

  int32_t n_cap = 0, C_max = 0;
  size_t ws_bytes = 0;
  CHECK_CKV(chunkkv_out_capacity(&p, &n_cap, &C_max));
  CHECK_CKV(chunkkv_workspace_size(&p, n_layers, n_reuse, &ws_bytes));
  const int groups = (n_layers + n_reuse - 1) / n_reuse;

  const void* q_d[64];
  const void* k_d[64];
  const void* v_d[64];
  void* ko_d[64];
  void* vo_d[64];
  const size_t out_bytes = (size_t)B * Hkv * n_cap * d * elt;
  for (int l = 0; l < n_layers; ++l) {
    char name[64];
    size_t nq = 0, nk = 0, nv = 0;
    void* hq = NULL;
    q_d[l] = NULL;
    if (l % n_reuse == 0) {
      snprintf(name, sizeof name, "q%d.bin", l);
      hq = read_file(dir, name, &nq);
      if (!hq) {
        fprintf(stderr, "cannot read %s\n", name);
        return 1;
      }
      void* dq;
      CHECK_CUDA(cudaMalloc(&dq, nq));
      CHECK_CUDA(cudaMemcpy(dq, hq, nq, cudaMemcpyHostToDevice));
      q_d[l] = dq;
      free(hq);
    }
    snprintf(name, sizeof name, "k%d.bin", l);
    void* hk = read_file(dir, name, &nk);
    snprintf(name, sizeof name, "v%d.bin", l);
    void* hv = read_file(dir, name, &nv);
    if (!hk || !hv) {
      fprintf(stderr, "cannot read the keys or values of layer %d\n", l);
      return 1;
    }
    void *dk, *dv, *dko, *dvo;
    CHECK_CUDA(cudaMalloc(&dk, nk));
    CHECK_CUDA(cudaMalloc(&dv, nv));
    CHECK_CUDA(cudaMalloc(&dko, out_bytes ? out_bytes : 16));
    CHECK_CUDA(cudaMalloc(&dvo, out_bytes ? out_bytes : 16));
    CHECK_CUDA(cudaMemcpy(dk, hk, nk, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, hv, nv, cudaMemcpyHostToDevice));
    free(hk);
    free(hv);
    k_d[l] = dk;
    v_d[l] = dv;
    ko_d[l] = dko;
    vo_d[l] = dvo;
  }
  const size_t idx_bytes = (size_t)groups * B * Hkv * (n_cap ? n_cap : 1) * sizeof(int32_t);
  const size_t cnt_bytes = (size_t)groups * B * Hkv * sizeof(int32_t);
  const size_t sc_bytes = (size_t)groups * B * Hkv * (C_max ? C_max : 1) * sizeof(float);
  void *d_idx, *d_cnt, *d_sc, *d_ws;
  CHECK_CUDA(cudaMalloc(&d_idx, idx_bytes));
  CHECK_CUDA(cudaMalloc(&d_cnt, cnt_bytes));
  CHECK_CUDA(cudaMalloc(&d_sc, sc_bytes));
  CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
  CHECK_CUDA(cudaMemset(d_ws, 0, ws_bytes));    /* the workspace starts zero-filled */

  CHECK_CKV(chunkkv_compress_layers(&p, n_layers, n_reuse, q_d, k_d, v_d, ko_d, vo_d, (int32_t*)d_idx,
                                    (int32_t*)d_cnt, (float*)d_sc, d_ws, ws_bytes, (chunkkv_stream_t)0));
  int32_t device_code = 0;
  CHECK_CKV(chunkkv_status_check(d_ws, (chunkkv_stream_t)0, &device_code));

  void* h = malloc(idx_bytes + cnt_bytes + sc_bytes + (out_bytes ? out_bytes : 16));
  if (!h) return 4;
  CHECK_CUDA(cudaMemcpy(h, d_cnt, cnt_bytes, cudaMemcpyDeviceToHost));
  if (!write_file(dir, "counts.bin", h, cnt_bytes)) return 5;
  CHECK_CUDA(cudaMemcpy(h, d_idx, idx_bytes, cudaMemcpyDeviceToHost));
  if (!write_file(dir, "indices.bin", h, idx_bytes)) return 5;
  CHECK_CUDA(cudaMemcpy(h, d_sc, sc_bytes, cudaMemcpyDeviceToHost));
  if (!write_file(dir, "scores.bin", h, sc_bytes)) return 5;
  for (int l = 0; l < n_layers; ++l) {
    char name[64];
    CHECK_CUDA(cudaMemcpy(h, ko_d[l], out_bytes, cudaMemcpyDeviceToHost));
    snprintf(name, sizeof name, "ko%d.bin", l);
    if (!write_file(dir, name, h, out_bytes)) return 5;
    CHECK_CUDA(cudaMemcpy(h, vo_d[l], out_bytes, cudaMemcpyDeviceToHost));
    snprintf(name, sizeof name, "vo%d.bin", l);
    if (!write_file(dir, name, h, out_bytes)) return 5;
  }
  snprintf(path, sizeof path, "%s/out_meta.txt", dir);
  FILE* of = fopen(path, "w");
  if (!of) return 5;
  fprintf(of, "%d %d\n", n_cap, C_max);
  fclose(of);
  free(h);
  for (int l = 0; l < n_layers; ++l) {
    cudaFree((void*)k_d[l]);
    cudaFree((void*)v_d[l]);
    cudaFree(ko_d[l]);
    cudaFree(vo_d[l]);
    if (q_d[l]) cudaFree((void*)q_d[l]);
  }
  cudaFree(d_idx);
  cudaFree(d_cnt);
  cudaFree(d_sc);
  cudaFree(d_ws);
  printf("compressed %d layers of %d sequences\n", n_layers, B);
  return 0;
}
