/*
 * pp.h -- C ABI of the GB300 layer-major batched int8 prefill library (libpp.so).
 *
 * What the library computes (sources are web pages on prompt prefill):
 *  - "Single-pass prefill" (SipLLM), section "The fix: batch over positions,
 *    stream each layer once": prefill(tokens, n, start_pos) inverts the loop
 *    nesting -- for each layer, read its weights once and sweep every prompt
 *    position through it; the causal K/V history kv[layer][0..i] is written
 *    position by position; only the last position's logits are produced,
 *    after a final RMSNorm and the output projection.
 *  - "Batched Prefill" (cellm), sections "The Solution", "What Stays
 *    Sequential", "Correctness": the projections become int8 GEMMs over a
 *    chunk of positions (weights read once per chunk), activations are
 *    quantised once per chunk and reused by every output row, attention is
 *    causal per position, and the chunked result equals the per-token path.
 *  - "Predictive prefetch" (SipLLM), section "The fix: an async double-buffer
 *    ring": in streamed mode layer L+1 is copied into the other ring slot
 *    while layer L computes; prefetch hits and misses are counted.
 *
 * Model: decoder-only transformer with RMSNorm, RoPE, grouped KV heads,
 * SwiGLU FFN, int8 per-output-row weights with f32 row scales, f32
 * embeddings, untied int8 output projection.
 *
 * Conventions for every entry point:
 *  - Return value: PP_OK (0) or a negative PP_ERR_* code. pp_last_error()
 *    gives a one-line description of the most recent failure on the calling
 *    thread.
 *  - "host" pointers are ordinary CPU memory; "device" pointers are CUDA
 *    global memory on the model's device. The caller owns every buffer it
 *    passes; the library never frees or retains them past the call, except
 *    where a function says otherwise.
 *  - A pp_model is used by one host thread at a time.
 *  - Nothing here falls back to the CPU: without a CUDA device every compute
 *    entry point fails with PP_ERR_CUDA.
 */
#ifndef PP_H
#define PP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define PP_OK 0
#define PP_ERR_ARG -1             /* null pointer, non-positive size, bad token id, unsupported shape */
#define PP_ERR_CAPACITY -2        /* start_pos + n exceeds the KV capacity max_seq */
#define PP_ERR_OOM -3             /* device or pinned-host allocation failed */
#define PP_ERR_CUDA -4            /* a CUDA runtime call failed (no device, launch error, ...) */
#define PP_ERR_DEVICE_TIMEOUT -5  /* a bounded device-side wait gave up; the kernel exited early */
#define PP_ERR_UNSUPPORTED -6     /* requested engine or mode is not available on this device */

/* ------------------------------------------------------------- constants */
#define PP_MODE_RESIDENT 0  /* every layer resident in HBM */
#define PP_MODE_STREAMED 1  /* layers in pinned host memory, streamed into a device ring */

/* Loop order of one prefill call ("Batched Prefill" section "The Solution":
 * chunks of the prompt swept through each layer; "Single-pass prefill":
 * stream each layer once for the whole prompt). Both give the same bits. */
#define PP_LOOP_CHUNK_OUTER 0 /* for each chunk, for each layer: scratch for max_chunk rows */
#define PP_LOOP_LAYER_OUTER 1 /* for each layer, for each chunk: every layer is fetched (streamed mode: copied
                                 from the host) once per call; keeps the residual stream of max_seq rows */

#define PP_GEMM_AUTO 0      /* fastest engine that passed its self-check on this device */
#define PP_GEMM_MMA 1       /* warp-level mma.sync s8 x s8 -> s32 */
#define PP_GEMM_TC 2        /* tcgen05 exact-integer GEMM (fp16 operands, f32 TMEM, int32 drain) */

/* Kernel classes that pp_config.profile_kernel can time with CUDA events. */
#define PP_KERNEL_NONE -1
#define PP_KERNEL_GEMM 0        /* all projection GEMMs */
#define PP_KERNEL_ATTENTION 1
#define PP_KERNEL_NORM_QUANT 2  /* RMSNorm + quantise and plain quantise */
#define PP_KERNEL_ROPE_KV 3
#define PP_KERNEL_LM_HEAD 4
#define PP_KERNEL_EMBED 5
#define PP_KERNEL_COUNT 6

/* Epilogues of pp_op_gemm (out is f32 [m][n] row-major, ldo = n unless stated). */
#define PP_EPI_STORE 0   /* out[t][r] = (float(acc) * w_scale[r]) * a_scale[t] */
#define PP_EPI_RESID 1   /* out[t][r] = out[t][r] + (float(acc) * w_scale[r]) * a_scale[t] */
#define PP_EPI_SWIGLU 2  /* rows interleaved in blocks of 16 (gate 16, up 16, ...):
                            out[t][16b+i] = silu(g) * u, out is [m][n/2] */

/* ------------------------------------------------------------------ model */
typedef struct pp_config {
  int32_t dim;          /* model width D */
  int32_t n_layers;
  int32_t n_heads;      /* query heads H */
  int32_t n_kv_heads;   /* KV heads Hkv, divides H */
  int32_t head_dim;     /* hd: 64 or 128 */
  int32_t ffn;          /* SwiGLU hidden width F, multiple of 16 */
  int32_t vocab;        /* V */
  float rms_eps;
  float rope_theta;
  int32_t max_seq;      /* KV capacity (positions); start_pos + n must not exceed it */
  int32_t max_chunk;    /* largest chunk any prefill call uses; sizes the activation scratch */
  int32_t mode;         /* PP_MODE_RESIDENT or PP_MODE_STREAMED */
  int32_t ring_slots;   /* streamed mode: 2 = double-buffer prefetch ring, 1 = synchronous single buffer */
  int32_t gemm_engine;  /* PP_GEMM_* */
  int32_t loop_order;   /* PP_LOOP_CHUNK_OUTER or PP_LOOP_LAYER_OUTER */
  int32_t profile_kernel; /* PP_KERNEL_* class to time with events around each launch, or PP_KERNEL_NONE */
  int32_t kv_grow;      /* 0: the K/V cache for max_seq positions is allocated at load; 1: only its address
                           range is reserved and device memory is mapped as calls write positions
                           ("Single-pass prefill": grow-on-demand KV), in steps of the device's allocation
                           granularity, and released by pp_kv_reset */
} pp_config;

/* Host weights (the pages' WeightSource seam: the math sees only these).
 * All matrices are int8 row-major [out][in] with one f32 scale per output row.
 * Per layer, in this order: wq [H*hd][D], wk [Hkv*hd][D], wv [Hkv*hd][D],
 * wo [D][H*hd], wg [F][D], wu [F][D], wd [D][F].
 * Read during pp_model_load only: in resident mode they are copied to the
 * device, in streamed mode into library-owned pinned host memory. */
typedef struct pp_weights {
  const float* tok_emb;          /* [vocab][D] f32 */
  const int8_t* const* w;        /* [n_layers * 7] matrices as above */
  const float* const* w_scale;   /* [n_layers * 7] row scales */
  const float* const* attn_norm; /* [n_layers] -> [D] RMSNorm gain before attention */
  const float* const* ffn_norm;  /* [n_layers] -> [D] RMSNorm gain before the FFN */
  const float* final_norm;       /* [D] */
  const int8_t* w_out;           /* [vocab][D] output projection */
  const float* w_out_scale;      /* [vocab] */
} pp_weights;

typedef struct pp_stats {
  int64_t calls;              /* prefill calls that completed */
  int64_t chunks;             /* chunks processed */
  int64_t tokens;             /* prompt positions processed */
  int64_t weight_bytes_read;  /* int8 weight + scale bytes the kernels fetch by design: every layer once
                                 per chunk, the output projection once per call ("Streamed" bytes) */
  int64_t h2d_bytes;          /* host-to-device bytes: token ids, and layer copies in streamed mode (once per
                                 layer per chunk chunk-outer, once per layer per call layer-outer) */
  int64_t prefetch_hits;      /* streamed mode: layer copy finished before the compute stream needed it */
  int64_t prefetch_misses;    /* streamed mode: compute waited on the copy (includes each call's first layer) */
  int64_t kernel_launches;    /* kernels this library launched */
  int64_t prof_launches;      /* launches of the profiled kernel class */
  double prof_ms;             /* summed event-timed duration of those launches */
  int64_t kv_bytes;           /* device memory backing the K/V cache now (a level, not a counter) */
  int64_t gemm_launches[5][6]; /* tcgen05 projection GEMM launches by [epilogue][tile]: epilogue 0 store,
                                  1 residual add, 2 SwiGLU, 3 raw int32, 4 QKV with RoPE and the K/V write;
                                  tile 0-2: chunks of more than 128 rows, 256 tokens x 256 / 192 / 128
                                  weight rows per CTA pair; tile 3-5: chunks of at most 128 rows, 256
                                  weight rows x 128 / 64 / 32 tokens */
} pp_stats;

typedef struct pp_model pp_model;

/* Create a model on the current CUDA device: validates cfg, repacks and
 * uploads (or pins) the weights, allocates the K/V cache for max_seq
 * positions, the activation scratch for max_chunk positions and the RoPE
 * table. On failure *out is NULL and nothing is leaked.
 * Errors: PP_ERR_ARG (bad cfg or null pointers), PP_ERR_OOM, PP_ERR_CUDA,
 * PP_ERR_UNSUPPORTED (gemm_engine not available). */
int pp_model_load(const pp_config* cfg, const pp_weights* w, pp_model** out);

/* Release all device and host memory of the model. NULL is a no-op. */
void pp_model_free(pp_model* m);

/* Layer-major prefill of host tokens[0..n) at positions start_pos ..
 * start_pos+n-1, `chunk` positions at a time (the last chunk may be ragged),
 * writing the last position's logits to host logits_out [vocab] f32.
 * Positions < start_pos must hold K/V from earlier calls (or be unused).
 * Synchronous: returns after logits_out is written.
 * Errors: PP_ERR_ARG (null, n <= 0, chunk <= 0 or > max_chunk, start_pos < 0,
 * token id outside [0, vocab)), PP_ERR_CAPACITY (start_pos + n > max_seq),
 * PP_ERR_CUDA, PP_ERR_DEVICE_TIMEOUT. On error logits_out is untouched and
 * K/V rows at positions >= start_pos are undefined. */
int pp_prefill(pp_model* m, const int32_t* tokens, int32_t n, int32_t start_pos, int32_t chunk,
               float* logits_out);

/* Same computation with device-resident ids d_tokens [n] and device output
 * d_logits [vocab], enqueued on `stream` (a cudaStream_t; NULL is the legacy
 * default stream, as for the pp_op_* calls) without host synchronisation:
 * work enqueued on `stream` afterwards (an event, a copy of d_logits) sees the
 * finished result. Each call is ordered after the model's previous call,
 * whatever stream that one was given (they share the K/V cache and scratch).
 * In streamed mode the layer copies run on the model's copy stream and the
 * compute on its own stream, joined to `stream` by events at both ends. Ids
 * are checked on the device: an id outside [0, vocab) gives a zero embedding
 * row and records PP_ERR_ARG in the model's device status, read by
 * pp_device_status(). */
int pp_prefill_device(pp_model* m, const int32_t* d_tokens, int32_t n, int32_t start_pos, int32_t chunk,
                      float* d_logits, void* stream);

/* The per-token path: pp_prefill(m, &token, 1, pos, 1, logits_out). */
int pp_forward_one(pp_model* m, int32_t token, int32_t pos, float* logits_out);

/* Wait for the model's streams and its last call (on whatever stream it was
 * enqueued) and return (and clear) the device status word: PP_OK, PP_ERR_ARG (bad id seen by pp_prefill_device) or
 * PP_ERR_DEVICE_TIMEOUT. */
int pp_device_status(pp_model* m);

/* Zero the whole K/V cache. */
int pp_kv_reset(pp_model* m);

/* Copy K (which = 0) or V (which = 1) rows [pos0, pos0+n_pos) of one layer to
 * host out [n_pos][n_kv_heads][head_dim] f32. */
int pp_kv_read(pp_model* m, int32_t layer, int32_t which, int32_t pos0, int32_t n_pos, float* out);

int pp_get_stats(const pp_model* m, pp_stats* out);
int pp_reset_stats(pp_model* m);

/* Select the kernel class (PP_KERNEL_*, or PP_KERNEL_NONE) whose launches are
 * bracketed by CUDA events on the launching stream from now on; their count
 * and summed duration appear in pp_stats (prof_launches, prof_ms). */
int pp_set_profile_kernel(pp_model* m, int32_t kernel_class);

/* Chunk overlap (1 on, 0 off; off after pp_model_load). The chunks of a call
 * rotate over min(32, chunks of the call) streams, each with its own scratch
 * set; a chunk waits, layer
 * by layer, only for the earlier chunks' K/V rows of that layer before its
 * attention reads them ("Single-pass prefill": K/V history written position
 * by position), so one chunk's kernels can use the SMs the others leave idle.
 * Chunk-outer order ("Batched Prefill") with resident weights: the chunks run
 * through their layers concurrently. Layer-outer order, resident or streamed:
 * the chunks of each layer run concurrently (streamed: every stream waits for
 * the layer's copy, and the ring slot is released after all of them). Results
 * are bit-identical to the serial order. This call allocates nothing: the
 * first prefill call that needs more streams than exist so far allocates the
 * missing scratch sets (each sized for max_chunk rows), streams and events
 * after waiting for the model's work, before it launches anything (PP_ERR_OOM
 * if that fails; what was made stays for later calls). Ignored while the
 * per-layer profile is on, for calls of a single chunk, and for streamed
 * weights in chunk-outer order. */
int pp_set_chunk_overlap(pp_model* m, int32_t enable);

/* CUDA graphs (1 on, 0 off; off after pp_model_load). With graphs on, the
 * first pp_prefill / pp_prefill_device call with a given (token and logits
 * buffers, n, start_pos, chunk, chunk overlap) is captured from the model's own
 * stream into an executable graph, which that call and every later identical
 * one launch as a whole on the caller's stream instead of launching each of
 * its kernels (thousands per call at small chunks) from the host. The graph
 * replays the same launches, so results and pp_stats are as without it.
 * Up to 8 graphs are kept per model (least recently used dropped first); off
 * frees them. Calls in streamed mode, with kv_grow, with a profiled kernel
 * class, with the per-layer profile or with a trace run launch by launch. */
int pp_set_graphs(pp_model* m, int32_t enable);

/* Per-layer stage profile ("Single-pass prefill", the per-layer profiler of
 * I/O and compute; "Predictive prefetch", the sync vs async loader A/B),
 * summed over every visit of the layer (one per chunk chunk-outer, one per
 * call layer-outer) since the last pp_reset_stats. */
typedef struct pp_layer_profile {
  double compute_ms;  /* first kernel of the visit to its last kernel, on the compute stream */
  double io_ms;       /* streamed mode: the layer's host-to-device copy on the copy stream */
  double wait_ms;     /* streamed mode: time the compute stream waited for that copy (prefetch misses) */
  int64_t visits;
} pp_layer_profile;

/* Turn the per-layer profile on (1) or off (0). It brackets every layer visit
 * with CUDA events (and every layer copy in streamed mode), which costs a few
 * microseconds per visit: keep it off in timed runs. */
int pp_set_layer_profile(pp_model* m, int32_t enable);

/* Copy the per-layer profile of the model's n_layers layers to out
 * [n_layers] (synchronises the model's streams first). */
int pp_get_layer_profile(const pp_model* m, pp_layer_profile* out, int32_t n_layers);

/* Record the residual stream at every layer boundary and the int8 codes at
 * every quantisation point (for layer-by-layer verification). While set,
 * each prefill call writes, for its positions p < max_pos:
 *  - d_x [(n_layers+1)][max_pos][dim] f32: the rows entering layer l at
 *    d_x[l][p], the rows leaving the last layer at d_x[n_layers][p];
 *  - d_codes [n_layers][4][max_pos][kmax] int8 with kmax = max(dim,
 *    n_heads*head_dim, ffn) and d_scales [n_layers][4][max_pos] f32: the
 *    codes and row scales of quantisation point q of layer l (0 attention
 *    input, 1 attention output, 2 FFN input, 3 SwiGLU output), each row
 *    starting at its kmax pitch (d_codes/d_scales may be NULL).
 * The caller owns the device buffers and keeps them alive while set; d_x
 * NULL switches tracing off. Calls whose positions exceed max_pos fail with
 * PP_ERR_CAPACITY while tracing is on. */
int pp_set_trace(pp_model* m, float* d_x, int8_t* d_codes, float* d_scales, int32_t max_pos);

/* The GEMM engine the model resolved to (PP_GEMM_MMA or PP_GEMM_TC). */
int pp_model_gemm_engine(const pp_model* m);

/* Static text for a status code. */
const char* pp_status_str(int status);
/* Description of the last failure on this thread ("" if none). */
const char* pp_last_error(void);

/* ------------------------------------------------- single steps (device) */
/* Each step of the hot path as its own entry point, on device pointers,
 * enqueued on `stream` (cudaStream_t; NULL = legacy default stream). They
 * run the same kernels, with the same launch shapes, as the model. Sizes
 * are checked on the host (PP_ERR_ARG); launch failures give PP_ERR_CUDA. */

/* Per-token absmax quantiser ("Batched Prefill", "The Solution": activations
 * quantised once per chunk). For each row t of x [rows][k] f32:
 * amax = max|x|, a_scale[t] = amax/127, q = clamp(rint_even(x * (127/amax)),
 * -127, 127) in f32; amax == 0 gives q = 0, a_scale = 0. Writes q8 [rows][k]
 * int8 and, if q16 is not NULL, the same codes as fp16 [rows][k]. */
int pp_op_quantize(const float* x, int32_t rows, int32_t k, int8_t* q8, uint16_t* q16, float* a_scale,
                   void* stream);

/* RMSNorm then quantise: y = x / sqrt(mean(x^2) + eps) * g (f32), then as
 * pp_op_quantize. If y_out is not NULL the normalised rows are written too. */
int pp_op_rmsnorm_quantize(const float* x, const float* g, int32_t rows, int32_t k, float eps, float* y_out,
                           int8_t* q8, uint16_t* q16, float* a_scale, void* stream);

/* Exact int8 GEMM: acc[t][r] = sum_i a[t][i] * w[r][i] as int32.
 * a8 [m][k] int8 (used by PP_GEMM_MMA), a16 [m][k] fp16 holding the same
 * integer codes (used by PP_GEMM_TC), w [n][k] int8. Needs k % 64 == 0 and
 * n % 32 == 0 (PP_GEMM_TC: n % 128 == 0). */
int pp_op_gemm_acc(int32_t engine, const int8_t* a8, const uint16_t* a16, const int8_t* w, int32_t m,
                   int32_t n, int32_t k, int32_t* acc, void* stream);

/* The same GEMM with its dequantising epilogue PP_EPI_* (f32, in the fixed
 * order (float(acc) * w_scale[r]) * a_scale[t]); out is f32, 16-byte aligned,
 * with leading dimension ldo (a multiple of 4); PP_GEMM_TC also needs 16-byte
 * aligned w_scale. */
int pp_op_gemm(int32_t engine, int32_t epilogue, const int8_t* a8, const uint16_t* a16, const int8_t* w,
               const float* w_scale, const float* a_scale, int32_t m, int32_t n, int32_t k, float* out,
               int32_t ldo, void* stream);

/* ------------------------------------------------------ host-buffer checks
 * The bit-exact steps on host buffers, for a caller without a device memory
 * library ("Batched Prefill", "Correctness": the batched GEMM is checked bit for
 * bit against per-token dot products). Each call copies its inputs into device
 * memory it allocates, runs the library's kernels on the legacy default stream,
 * waits for them, copies the results into the caller's buffers and frees what it
 * allocated. Every pointer is caller-owned host memory; nothing is kept after the
 * call. The GEMMs run on the tcgen05 engine when n % 128 == 0 and on the mma.sync
 * engine otherwise (both give the same bits). Errors: PP_ERR_ARG (a null
 * pointer, a size <= 0, k % 4 for the quantiser, k % 64 or n % 32 for the GEMMs),
 * PP_ERR_OOM, PP_ERR_CUDA, PP_ERR_DEVICE_TIMEOUT (a bounded wait of the tcgen05
 * GEMM gave up). After an error the outputs are untouched. */

/* pp_op_quantize on host rows: x [rows][k] f32 in; q [rows][k] int8 and
 * a_scale [rows] f32 out. */
int pp_debug_quantize(const float* x, int32_t rows, int32_t k, int8_t* q, float* a_scale);

/* acc[t][r] = sum_i a[t][i] * w[r][i] as int32: a [m][k], w [n][k] int8 in,
 * acc [m][n] int32 out. */
int pp_debug_gemm_i8(const int8_t* a, const int8_t* w, int32_t m, int32_t n, int32_t k, int32_t* acc);

/* The dequantising epilogue on the same GEMM: out[t][r] =
 * (float(acc[t][r]) * w_scale[r]) * a_scale[t], then, if resid is not NULL,
 * out[t][r] = resid[t][r] + out[t][r] (the residual epilogue), all in f32 with
 * round-to-nearest. w_scale [n], a_scale [m], resid and out [m][n] f32. */
int pp_debug_gemm_epilogue(const int8_t* a, const int8_t* w, const float* w_scale, const float* a_scale,
                           const float* resid, int32_t m, int32_t n, int32_t k, float* out);

/* K-extent of one exact f32 accumulation segment of the tcgen05 engine
 * (process-wide; default and maximum 1024, multiple of 64). Partial sums of
 * up to 1024 products of int8 values stay below 2^24 and are exact in f32;
 * shorter segments only add drains. Errors: PP_ERR_ARG out of range. */
int pp_set_exact_segment(int32_t seg_k);

/* ---------------------------------------------------------------- test hooks
 * Failure paths made on purpose without faulting the GPU (the pages' only
 * failure handling is graceful degradation: a prefetch miss blocks until the
 * copy is ready, "Predictive prefetch"). */

/* Run the tcgen05 GEMM (int32 result into acc, as pp_op_gemm_acc) with its MMA
 * issuer held back and every mbarrier wait bounded by wait_us microseconds:
 * nothing completes the accumulators, so every other role's bounded wait runs
 * out, records the timeout, lets its copies land, frees its tensor memory and
 * exits. Synchronous. Returns PP_ERR_DEVICE_TIMEOUT when the kernel reported
 * the timeout (the expected result), PP_OK if it did not, or an argument /
 * CUDA error. The device stays usable afterwards. */
int pp_debug_gemm_stall(int32_t wait_us, const uint16_t* a16, const int8_t* w, int32_t m, int32_t n, int32_t k,
                        int32_t* acc);

/* Streamed-mode loader fault: 0 none; 1 the ring issues no prefetch, so every
 * layer copy starts only when its visit begins (every visit a miss; results
 * unchanged). Errors: PP_ERR_ARG. */
int pp_debug_loader_fault(pp_model* m, int32_t fault);

/* Process-wide cap on the device bytes one model may hold (its allocations at
 * load plus the grown K/V cache); 0 removes the cap. A load or a K/V growth
 * that would pass it fails with PP_ERR_OOM and leaks nothing. */
int pp_debug_alloc_cap(int64_t bytes);

/* Status of the single-step GEMM calls on the tcgen05 engine (pp_op_gemm,
 * pp_op_gemm_acc, pp_op_gemm_noalloc) on the current device. Every mbarrier
 * wait inside those kernels is bounded; when one runs out the kernel records
 * it in a device status word that all these calls share, lets its copies land
 * and exits early, leaving its output incomplete. This call waits for `stream`
 * (cudaStream_t; NULL = legacy default stream), then returns PP_OK, or
 * PP_ERR_DEVICE_TIMEOUT (and clears the word) if any such call timed out since
 * the last query. The word lives in the library's own device memory. */
int pp_op_status(void* stream);

/* Test hook: from now on every single-step tcgen05 GEMM call holds back its MMA
 * issuer and bounds each mbarrier wait by wait_us microseconds, so every call
 * times out on purpose (pp_op_status then reports PP_ERR_DEVICE_TIMEOUT) without
 * faulting or hanging the GPU; wait_us = 0 restores normal calls. Process-wide.
 * Errors: PP_ERR_ARG (wait_us < 0). */
int pp_debug_op_stall(int32_t wait_us);

/* Capacity of the fixed scratch of pp_op_gemm_noalloc, per device. */
#define PP_NOALLOC_PART_BYTES (32 * 1024 * 1024) /* partial int32 tiles */
#define PP_NOALLOC_COUNTERS 4096                 /* per-tile arrival counters */

/* The tcgen05 GEMM of pp_op_gemm (engine PP_GEMM_TC) without any device
 * allocation, for callers that may not allocate device memory while they run
 * (an application whose device memory is all held by its own pool allocator,
 * or a latency-critical loop where cudaMalloc/cudaFree would block or
 * synchronise the device). The pages have no counterpart: it only changes
 * where the GEMM's stream-K scratch lives.
 * The scratch (partial int32 tiles of GEMMs with few output tiles and long K,
 * and their arrival counters) is a fixed array inside the library:
 * PP_NOALLOC_PART_BYTES plus PP_NOALLOC_COUNTERS counters, placed on every
 * device that loads the library's device code and kept until the process
 * exits, whether or not this function is ever called. It is not counted by
 * pp_debug_alloc_cap nor in any model's memory figures. Shapes whose plan needs
 * more (pp_op_gemm_noalloc_need; e.g. m = 1024, n = 4096, k = 14336 on a GB300)
 * fail with PP_ERR_ARG and a message naming both sizes; shapes that need no
 * scratch always run.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process, so make that
 * first call before any stream capture, and do not reset the device
 * (cudaDeviceReset) after it.
 * All calls on a device share its one array, which keeps the last call's
 * contents (the counters are cleared on `stream` at the start of every call):
 * calls on the same device whose executions overlap, for example on two
 * streams, race and give wrong results. A bounded wait that runs out is
 * reported by pp_op_status. Arguments and errors as pp_op_gemm, with a16, w and
 * w_scale 16-byte aligned. */
int pp_op_gemm_noalloc(int32_t epilogue, const uint16_t* a16, const int8_t* w, const float* w_scale,
                       const float* a_scale, int32_t m, int32_t n, int32_t k, float* out, int32_t ldo, void* stream);

/* Scratch that pp_op_gemm_noalloc (and pp_op_gemm on the tcgen05 engine) plans
 * for an m x n x k GEMM on the current device: partial-tile bytes and counters
 * (both 0 when it runs whole tiles; the plan depends on the device's SM count).
 * Errors: PP_ERR_ARG (k % 64, n % 128), PP_ERR_UNSUPPORTED (no sm_103 device). */
int pp_op_gemm_noalloc_need(int32_t m, int32_t n, int32_t k, int64_t* part_bytes, int64_t* counters);

/* Test hook: set every arrival counter of the fixed scratch on the current
 * device to `value` (synchronous), as a call that gave up part of the way would
 * leave them. pp_op_gemm_noalloc clears what it uses, so its results do not
 * change. */
int pp_debug_noalloc_poison(int32_t value);

/* RoPE + K/V write for `rows` positions start_pos..: qkv [rows][(H+2Hkv)*hd]
 * f32 (q heads, then k heads, then v heads) -> q_out [rows][H][hd] rotated,
 * k rotated into k_cache[start_pos+i], v copied into v_cache[start_pos+i]
 * (caches [*][Hkv][hd] f32). Pairs (j, j+hd/2) turn by pos*theta^(-2j/hd).
 * rope_table [max_pos][hd/2][2] (cos, sin) comes from pp_op_rope_table. */
int pp_op_rope_kv(const float* qkv, int32_t rows, int32_t start_pos, int32_t n_heads, int32_t n_kv_heads,
                  int32_t head_dim, const float* rope_table, float* q_out, float* k_cache, float* v_cache,
                  void* stream);

/* Fill rope_table [max_pos][hd/2][2] with cos/sin of pos*theta^(-2j/hd)
 * (angles in double, rounded to f32). */
int pp_op_rope_table(int32_t max_pos, int32_t head_dim, float theta, float* rope_table, void* stream);

/* Causal attention ("Single-pass prefill": position i attends over
 * kv[0..i]): q [rows][H][hd] at positions start_pos+i, k/v caches
 * [*][Hkv][hd]; o [rows][H][hd] = softmax((q.k_j)/sqrt(hd), j <= pos) v.
 * Query head h reads KV head h / (H / Hkv). f32 on CUDA cores; every
 * query's reduction order depends only on its absolute position (keys are
 * reduced in ranges of 512 at fixed positions, then the ranges in order).
 * When start_pos + rows > 512 the call uses a library-owned device
 * workspace, grown on first need (that growth synchronises the device) and
 * shared by all calls: calls on different streams must not overlap. */
int pp_op_attention(const float* q, const float* k_cache, const float* v_cache, int32_t rows, int32_t start_pos,
                    int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float* o, void* stream);

/* Output projection of one quantised row: logits[v] = (float(sum_i q8[i] *
 * w_out[v][i]) * w_scale[v]) * a_scale[0], for v < vocab. */
int pp_op_lm_head(const int8_t* q8, const float* a_scale, const int8_t* w_out, const float* w_scale,
                  int32_t vocab, int32_t dim, float* logits, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PP_H */
