/*
 * chunkkv.h - ChunkKV chunk-level KV-cache compression on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the one of "ChunkKV: Semantic-Preserving KV Cache
 * Compression for Efficient Long-Context LLM Inference" (NeurIPS'25 notes):
 *   §4.1 Algorithm 1  - score every key against an observation window of the
 *                       last w queries, sum the scores per chunk of c tokens,
 *                       keep the top k = floor(L_max / c) chunks plus the last
 *                       w tokens, index_select K and V by the kept positions;
 *   §4.2 Algorithm 2  - layers with l mod N_reuse != 0 do not score; they
 *                       gather with the index list of layer
 *                       floor(l / N_reuse) * N_reuse.
 * The window scores are attention probabilities as in "Kara" §2 Eq. (1):
 * softmax over all T keys of (Q_w K^T / sqrt(d)) for each window-query row,
 * summed over the w window rows and over the G = Hq / Hkv query heads that
 * share a KV head (query head hq belongs to KV head hq / G).  By default no
 * causal mask applies inside the window (the algorithm as printed);
 * chunkkv_params.causal_window = 1 masks each window query to the keys at or
 * before its own position.  Top-k ties go to the lower chunk index.
 * The kept list is the ascending, duplicate-free union of the selected
 * chunks' tokens and the last w tokens.
 *
 * Conventions for every call
 *  - Device pointers point to GPU global memory owned by the caller; the
 *    library never allocates or frees device memory while it runs and keeps
 *    no per-call state between calls (its one fixed device array is the
 *    scratch of chunkkv_score_noalloc, described there).  Host arrays
 *    (cu_seqlens, pointer tables) are read during the call only.
 *  - "Addressable" pointers (the K/V data that only the gather and the
 *    portable scoring kernel touch, marked below) may also point to host
 *    memory that the GPU reads and writes directly: pinned (cudaHostAlloc,
 *    cudaHostRegister) or, on systems with coherent host access, any host
 *    memory.  The kernels then move only the kept rows across the host link
 *    (NVLink-C2C on Grace systems) instead of a staging copy of whole
 *    layers.  Keys read by the tensor-core scoring kernel go through a TMA
 *    tensor map and must be device memory (cudaMalloc or a stream-ordered
 *    pool; cudaPointerGetAttributes type cudaMemoryTypeDevice); a host or
 *    managed pointer there is rejected with CHUNKKV_ERR_INVALID_ARG before
 *    anything is launched.
 *  - Every call is asynchronous on the given stream (0 = legacy default).
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns an error code and launches nothing.  A failed launch
 *    returns CHUNKKV_ERR_CUDA.  Conditions the GPU detects (a pipeline wait
 *    that ran out of time) are recorded in the workspace and reported by
 *    chunkkv_status_check.
 *  - Layouts (elements; the head dimension d is always contiguous):
 *      q_win        [B, w, Hq, d]  at q_win[b*q_stride_b + i*q_stride_w + hq*q_stride_h + e]
 *      k, v         [T_total, Hkv, d] at x[t*kv_stride_t + h*kv_stride_h + e], sequence b
 *                   owning rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (varlen, ragged)
 *      chunk_scores [B, Hkv, C_max] fp32, chunk i of sequence b at [b][h][i], i < C_b
 *      indices      [B, Hkv, n_cap_max] int32, positions local to the sequence
 *      counts       [B, Hkv] int32
 *      k_out, v_out [B, Hkv, n_cap_max, d] in the input dtype
 *    Rows at or beyond counts[b][h] of indices / k_out / v_out, and chunk
 *    scores at or beyond C_b, are left unwritten.
 *  - Alignment: q_win, k, v, k_out and v_out start on 16-byte boundaries, and
 *    kv_stride_t, kv_stride_h, q_stride_* and d are multiples of 16 bytes.
 */
#ifndef CHUNKKV_H_
#define CHUNKKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* chunkkv_stream_t;   /* the same type as cudaStream_t */

typedef enum chunkkv_status {
  CHUNKKV_OK = 0,
  CHUNKKV_ERR_INVALID_ARG = 1,         /* a size, pointer, stride or alignment is invalid   */
  CHUNKKV_ERR_UNSUPPORTED = 2,         /* valid, but outside what this build implements    */
  CHUNKKV_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < chunkkv_workspace_size(...)            */
  CHUNKKV_ERR_CUDA = 4,                /* a CUDA runtime call or kernel launch failed        */
  CHUNKKV_ERR_TIMEOUT = 5              /* a device-side wait gave up (chunkkv_status_check) */
} chunkkv_status;

typedef enum chunkkv_dtype { CHUNKKV_F32 = 0, CHUNKKV_BF16 = 1 } chunkkv_dtype;

/* Largest batch one call accepts (the sequence table travels as a launch argument). */
#define CHUNKKV_MAX_BATCH 1024
/* Largest number of layers one chunkkv_gather call moves. */
#define CHUNKKV_MAX_GATHER_LAYERS 64

typedef struct chunkkv_params {
  int32_t B;        /* sequences, 0 <= B <= CHUNKKV_MAX_BATCH                                  */
  int32_t Hq;       /* query heads; Hq % Hkv == 0                                               */
  int32_t Hkv;      /* key/value heads, >= 1                                                    */
  int32_t d;        /* head dimension, 1..256                                                   */
  int32_t w;        /* observation window = number of window queries = recent tokens kept, >= 0 */
  int32_t c;        /* chunk size, >= 1                                                         */
  int32_t L_max;    /* compressed budget; k = min(L_max / c, C_b) chunks per (b, head), >= 0     */
  int32_t dtype;    /* chunkkv_dtype of q_win, k, v, k_out, v_out                                */
  const int32_t* cu_seqlens;  /* HOST array [B+1]: cu[0] = 0, non-decreasing; T_b = cu[b+1]-cu[b] */
  int64_t q_stride_b, q_stride_w, q_stride_h;   /* element strides of q_win                     */
  int64_t kv_stride_t, kv_stride_h;             /* element strides of k and v (and their layers) */
  int32_t causal_window;  /* 0: every window query sees all T_b keys (the algorithm as printed);
                             1: window query q (0 <= q < w) sits at position T_b - w + q and sees
                             keys 0 .. T_b - w + q only (a query at a negative position adds nothing) */
} chunkkv_params;

/*
 * Output capacities: n_cap_max = max_b min(T_b, k_b*c + min(w, T_b)) is the row
 * capacity per (b, head) of indices/k_out/v_out; C_max = max_b ceil(T_b / c) is
 * the chunk capacity of chunk_scores.  Either output pointer may be NULL.
 */
chunkkv_status chunkkv_out_capacity(const chunkkv_params* p, int32_t* n_cap_max, int32_t* C_max);

/*
 * Bytes of device workspace chunkkv_score / chunkkv_compress_layers need for
 * these shapes (n_layers, n_reuse as passed to chunkkv_compress_layers; use
 * 1, 1 for chunkkv_score).  The workspace must be zero-filled before its first
 * use (cudaMemset / torch.zeros); afterwards the library keeps it consistent.
 * Its first 256 bytes hold the device error word (chunkkv_status_check) and the
 * counter from which the CTAs of a tensor-core scoring launch claim their work
 * items; the launch leaves the counter at zero when it ends.
 * One workspace must not be used by two calls that can run at the same time.
 */
chunkkv_status chunkkv_workspace_size(const chunkkv_params* p, int32_t n_layers, int32_t n_reuse,
                                      size_t* bytes);

/*
 * Window scores per chunk for one layer (ChunkKV §4.1 Algorithm 1 steps 1-3,
 * with the probabilities of Kara §2 Eq. (1)):
 *   A[b][h][i] = sum over g < G, q < w, j in chunk i of softmax_j(Q_w[b,q,h*G+g,:] . K[b,j,h,:] / sqrt(d))
 * q_win: addressable (on the tensor-core path device Q_w is read through a
 * tensor map when w divides 128, host Q_w is first packed with plain loads);
 * k: device when chunkkv_score_path(p) is 1 (tensor cores), else addressable;
 * layouts above.  chunk_scores: device, written for
 * i < C_b.  ws: device workspace of ws_bytes >= chunkkv_workspace_size(p, 1, 1).
 */
chunkkv_status chunkkv_score(const chunkkv_params* p, const void* q_win, const void* k,
                             float* chunk_scores, void* ws, size_t ws_bytes, chunkkv_stream_t stream);

/*
 * Top-k chunk selection and kept-index construction (ChunkKV §4.1 Algorithm 1
 * steps 4-6): for each (b, h) keep the k_b = min(L_max / c, C_b) chunks of
 * largest chunk_scores (ties to the lower chunk index; -0.0 equals +0.0; the
 * scores must not be NaN), and write the ascending union of their tokens and
 * of the last w tokens to indices[b][h][0 .. counts[b][h]).
 * chunk_scores: device [B, Hkv, C_max]; indices, counts: device outputs.
 */
chunkkv_status chunkkv_select(const chunkkv_params* p, const float* chunk_scores, int32_t* indices,
                              int32_t* counts, chunkkv_stream_t stream);

/*
 * index_select of K and V by a kept-index list (ChunkKV §4.1 Algorithm 1 step
 * 6), for n_layers layers that share one list (ChunkKV §4.2 Algorithm 2):
 *   k_out[l][b][h][r][:] = k[l][cu_seqlens[b] + indices[b][h][r]][h][:]  for r < counts[b][h]
 * and the same for v.  k, v, k_out, v_out: HOST arrays of n_layers
 * addressable pointers (1 <= n_layers <= CHUNKKV_MAX_GATHER_LAYERS); indices,
 * counts: device.
 * Indices must lie in [0, T_b); the copy is bit-exact.
 */
chunkkv_status chunkkv_gather(const chunkkv_params* p, int32_t n_layers, const int32_t* indices,
                              const int32_t* counts, const void* const* k, const void* const* v,
                              void* const* k_out, void* const* v_out, chunkkv_stream_t stream);

/*
 * The whole path over n_layers layers (ChunkKV §4.2 Algorithm 2 around §4.1
 * Algorithm 1): layers with l % n_reuse == 0 run score + select into index
 * group g = l / n_reuse; every layer l gathers its own K, V with group
 * l / n_reuse.
 *   q_win: HOST array of n_layers addressable pointers (entries of layers
 *          with l % n_reuse != 0 are not read and may be NULL; as for
 *          chunkkv_score, host Q_w costs one packing launch);
 *   k, v, k_out, v_out: HOST arrays of n_layers addressable pointers, except
 *          that k[l] of a scoring layer (l % n_reuse == 0) is device memory
 *          when chunkkv_score_path(p) is 1;
 *   indices: device [ceil(n_layers / n_reuse), B, Hkv, n_cap_max];
 *   counts:  device [ceil(n_layers / n_reuse), B, Hkv];
 *   chunk_scores: NULL, or device [ceil(n_layers / n_reuse), B, Hkv, C_max];
 *   ws: device workspace of ws_bytes >= chunkkv_workspace_size(p, n_layers, n_reuse).
 */
chunkkv_status chunkkv_compress_layers(const chunkkv_params* p, int32_t n_layers, int32_t n_reuse,
                                       const void* const* q_win, const void* const* k,
                                       const void* const* v, void* const* k_out, void* const* v_out,
                                       int32_t* indices, int32_t* counts, float* chunk_scores,
                                       void* ws, size_t ws_bytes, chunkkv_stream_t stream);

/*
 * Incremental compression during decoding (the notes keep the compressed cache
 * through decoding, ChunkKV §5.6; Kara §2 Eqs. (2)-(3) compress again once the
 * cache reaches its threshold), over n_layers layers with the index reuse of
 * ChunkKV §4.2 Algorithm 2.  Sequence b of p is the current cache of one
 * sequence: its first n_prev[b] positions were kept by earlier passes, the
 * rest are the n_new = T_b - n_prev[b] tokens decoded since.  A scoring layer
 * (l % n_reuse == 0) re-scores the new tail only (ChunkKV §4.1 Algorithm 1 on
 * the tail), with every window row normalised over all T_b keys of the cache:
 *   A[g][b][h][i] = sum over g', q and tail tokens j in chunk i of softmax over all T_b keys,
 * chunk i being tail tokens [i*c, min(i*c + c, n_new)); it keeps the
 * min(L_max / c, ceil(n_new / c)) best tail chunks (ties to the lower index)
 * plus the last w tail tokens into index group g = l / n_reuse, and every
 * layer l gathers its own rows with group l / n_reuse:
 *   indices[g][b][h][r]: ascending TAIL positions (0 = the first token after
 *                        the kept prefix), r < counts[g][b][h];
 *   k_out[l][b][h][r][:] = k[l][cu_seqlens[b] + n_prev[b] + indices[l / n_reuse][b][h][r]][h][:],
 *                        same for v,
 * which the caller appends after the n_prev[b] rows it keeps.  L_max is the
 * budget for the tail of this pass; n_prev is the same for every layer (the
 * layers' caches grow together).  The prefix positions are never selected or
 * moved.  Caches of different KV heads usually differ in length after a pass:
 * pass each head's cache as a sequence of its own (Hkv = 1, its G query heads)
 * when they do.
 *   n_prev: HOST [B], 0 <= n_prev[b] <= T_b;
 *   q_win, k, v, k_out, v_out: HOST arrays of n_layers pointers as for
 *          chunkkv_compress_layers; k_out[l], v_out[l] [B, Hkv, n_cap_max, d] with
 *          n_cap_max from chunkkv_tail_sizes;
 *   indices: device [ceil(n_layers / n_reuse), B, Hkv, n_cap_max];
 *   counts:  device [ceil(n_layers / n_reuse), B, Hkv];
 *   chunk_scores: NULL, or device [ceil(n_layers / n_reuse), B, Hkv, C_max] (tail
 *          chunks; entries >= C_b unspecified);
 *   ws: device workspace of ws_bytes >= chunkkv_tail_sizes' ws_bytes for the same
 *       n_layers and n_reuse (zero-filled before its first use, like
 *       chunkkv_workspace_size's).
 * B may be at most CHUNKKV_MAX_BATCH / 2 (the prefix and the tail of each cache
 * are scored as two sequences); causal_window must be 0 (CHUNKKV_ERR_UNSUPPORTED).
 */
chunkkv_status chunkkv_tail_sizes(const chunkkv_params* p, const int32_t* n_prev, int32_t n_layers, int32_t n_reuse,
                                  int32_t* n_cap_max, int32_t* C_max, size_t* ws_bytes);
chunkkv_status chunkkv_compress_tail(const chunkkv_params* p, const int32_t* n_prev, int32_t n_layers, int32_t n_reuse,
                                     const void* const* q_win, const void* const* k, const void* const* v,
                                     void* const* k_out, void* const* v_out, int32_t* indices, int32_t* counts,
                                     float* chunk_scores, void* ws, size_t ws_bytes, chunkkv_stream_t stream);

/*
 * Window scores for callers that cannot allocate device memory.  The ChunkKV
 * notes have no counterpart for this call; it exists for code that must not
 * call cudaMalloc when it scores (code running inside a memory pool or arena
 * that owns all device memory, allocator callbacks, runtimes with a memory
 * budget fixed at start-up) and has no workspace to lend.
 * It computes exactly what chunkkv_score computes, with the portable scoring
 * kernel, and takes no workspace: its scratch is one device array of
 * CHUNKKV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.  It allocates nothing.
 *  - Shapes whose scratch would exceed that array return
 *    CHUNKKV_ERR_WORKSPACE_TOO_SMALL before anything is launched (about
 *    4 * w * G * Hkv * sum_b T_b / c bytes are needed; e.g. T = 32768 tokens with
 *    w*G = 128 rows and 8 KV heads fits).
 *  - All calls share the array and it keeps the last call's contents; a call
 *    reads only what it wrote itself, so nothing has to be cleared.  Calls whose
 *    kernels can overlap on the GPU (other streams, other threads) race on it.
 *  - The first call on each device looks up the array's device address with
 *    that device current; make it before any stream capture begins.
 */
#define CHUNKKV_NOALLOC_SCRATCH_BYTES (16u << 20)
chunkkv_status chunkkv_score_noalloc(const chunkkv_params* p, const void* q_win, const void* k,
                                     float* chunk_scores, chunkkv_stream_t stream);

/*
 * Synchronises the stream, then reads and clears the device-side error word of
 * the workspace.  Returns CHUNKKV_ERR_TIMEOUT if a kernel gave up waiting since
 * the last check (device_code, if not NULL, receives the raw code: the site
 * that gave up), CHUNKKV_ERR_CUDA if the stream reported an error, else CHUNKKV_OK.
 */
chunkkv_status chunkkv_status_check(void* ws, chunkkv_stream_t stream, int32_t* device_code);

/*
 * Adjacent-layer overlap of kept index lists: the Jaccard similarity of
 * consecutive layers' selections that ChunkKV §4.2 reports as the observation
 * behind Algorithm 2 (layer-wise index reuse), as exact counts.  Run on lists
 * scored independently per layer (chunkkv_compress_layers with n_reuse = 1) it
 * measures how much a reuse depth N_reuse would change the kept tokens.
 *   indices: device [n_lists, B, Hkv, n_cap_max] int32, each list ascending and
 *            duplicate-free in [0, T_b) for its first counts[...] entries
 *            (the layout chunkkv_compress_layers writes);
 *   counts:  device [n_lists, B, Hkv] int32;
 *   inter, uni: device [n_lists - 1, B, Hkv] int32, written with
 *            |I_l ∩ I_{l+1}| and |I_l ∪ I_{l+1}| for l = 0 .. n_lists - 2
 *            (Jaccard = inter / uni; two empty lists give 0 / 0).
 * Positions outside [0, T_b) are ignored.  n_lists == 1 or an empty batch
 * writes nothing.  Returns CHUNKKV_ERR_UNSUPPORTED when a sequence is longer
 * than the kernel's shared-memory bitmap holds (about 1.86 M tokens).
 */
chunkkv_status chunkkv_layer_overlap(const chunkkv_params* p, int32_t n_lists, const int32_t* indices,
                                     const int32_t* counts, int32_t* inter, int32_t* uni, chunkkv_stream_t stream);

/*
 * Self test of the failure path (a test aid; no counterpart in the pages).
 * Launches one thread that first starts an asynchronous bulk copy of ws bytes
 * 128..191 into shared memory, then waits, through the same bounded wait as the
 * tensor-core scoring kernel, on a barrier that nothing completes.  The wait
 * gives up after about a millisecond and records device code 0x1FF in the error
 * word of ws; the thread then drains its copy as the scoring kernel's teardown
 * does after a give-up (a bounded wait on the copy's own barrier phase, never a
 * fixed pause) and writes the 64 bytes that landed to ws bytes 64..127.  The
 * kernel returns and leaves the context usable; a following
 * chunkkv_status_check(ws, ...) returns CHUNKKV_ERR_TIMEOUT with that code.
 *   ws: device workspace of at least 256 bytes (bytes 0..3 and 64..127 are written).
 * Returns CHUNKKV_ERR_INVALID_ARG for a NULL, misaligned or too small ws.
 */
chunkkv_status chunkkv_selftest_wait_timeout(void* ws, size_t ws_bytes, chunkkv_stream_t stream);

/*
 * Throughput probe of the exponential unit (a measurement aid; no counterpart in
 * the pages).  The scoring kernels evaluate one base-2 exponential
 * (ex2.approx.ftz.f32) per window logit; this call launches `blocks` CTAs of
 * CHUNKKV_PROBE_THREADS threads, each thread evaluating `iters` rounds of
 * CHUNKKV_PROBE_CHAINS independent exponentials of that instruction, i.e.
 * blocks * CHUNKKV_PROBE_THREADS * CHUNKKV_PROBE_CHAINS * iters of them in all.
 * Timing the call (events on `stream`) gives the exponential rate that bounds
 * the scoring phase.
 *   sink: device, blocks * CHUNKKV_PROBE_THREADS floats (one result per thread).
 * Returns CHUNKKV_ERR_INVALID_ARG for a NULL sink or a non-positive count.
 */
#define CHUNKKV_PROBE_THREADS 256
#define CHUNKKV_PROBE_CHAINS 16
chunkkv_status chunkkv_probe_ex2(float* sink, int32_t blocks, int32_t iters, chunkkv_stream_t stream);

/* Static description of a status code. */
const char* chunkkv_status_string(chunkkv_status s);

/* Which scoring kernel chunkkv_score would use for these shapes: 0 = SIMT, 1 = tensor-core. */
int32_t chunkkv_score_path(const chunkkv_params* p);

/*
 * Number of CUDA kernels this process has launched through the library so far
 * (every entry point, every device and host thread; a relaxed atomic counter
 * that only grows).  The difference of two readings around a region counts the
 * library's kernel launches in it.  Never fails.
 */
uint64_t chunkkv_launch_count(void);

/*
 * Phase timing of chunkkv_compress_layers and chunkkv_compress_tail (a
 * measurement aid).
 *   events: HOST array of CHUNKKV_PHASE_EVENTS cudaEvent_t handles (as void*)
 *           that the caller created and keeps alive; NULL with n_events = 0
 *           switches recording off.
 * While set, each chunkkv_compress_layers or chunkkv_compress_tail call made
 * by the same host thread records events[i] on its stream at phase boundary i:
 * 0 before the window-row packing (a phase without a launch when the scoring
 * kernel reads the window rows from q_win itself: w divides 128), 1 before
 * scoring, 2 before the log-sum-exp, 3 before the finalisation (for token-level
 * chunks in two passes: the second pass and the sum of its partial arrays), 4
 * before the top-k selection, 5 before the gather, 6 after the gather.  When
 * one kernel takes the log-sum-exp, the finalisation and the selection (calls
 * with enough (group, sequence, head) triples to fill the GPU), boundaries 2
 * and 3 come before it and 4 after it, so its time shows as the
 * finalisation's.  A record between two launches ends the
 * programmatic-dependent-launch overlap there, so recorded calls run a little
 * slower than unrecorded ones.
 * Returns CHUNKKV_ERR_INVALID_ARG if n_events is neither 0 nor
 * CHUNKKV_PHASE_EVENTS or a handle is NULL (the previous setting then stays).
 */
#define CHUNKKV_PHASE_EVENTS 7
chunkkv_status chunkkv_set_phase_events(void* const* events, int32_t n_events);

#ifdef __cplusplus
}
#endif

#endif /* CHUNKKV_H_ */
