/*
 * CPU oracle of layer-major batched int8 prefill -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct C implementation of what the prefill
 * path computes. Only the tests, the package's smoke check and the bench's
 * CPU-baseline leg may call it; the CUDA library never links, loads or
 * calls anything here, and this file includes nothing from it.
 *
 * Sources (web pages on prompt prefill):
 *  - "Single-pass prefill" (SipLLM), section "The fix: batch over positions,
 *    stream each layer once": the loop order (for each layer, sweep every
 *    prompt position through it), the causal K/V history written position
 *    by position, and last-position-only logits after a final RMSNorm.
 *  - "Batched Prefill" (cellm), sections "The Solution", "What Stays
 *    Sequential" and "Correctness": int8 projections as GEMMs over a chunk
 *    of positions, activations quantised once per chunk and reused by every
 *    output row, threads split by weight rows, attention per position, and
 *    chunked output identical to the per-token path.
 *  - The measured model configurations: RMSNorm (eps), RoPE (theta),
 *    SwiGLU FFN, grouped KV heads, int8 per-output-row weights with f32 row
 *    scales, f32 embeddings.
 *
 * Precision: integer GEMMs are exact int32. The activation quantiser and
 * the dequantising epilogue float(acc) * w_scale * a_scale are f32 in that
 * fixed order, because the method fixes them. Everything else (RMSNorm,
 * RoPE, attention softmax, SiLU) is computed in double and rounded to f32
 * where the result is stored (residual stream, K/V cache, activations).
 */
#ifndef PP_ORACLE_H
#define PP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab, max_seq;
  float rms_eps, rope_theta;
} orc_config;

/* Host weights, borrowed for the model's lifetime. Matrices are int8
 * row-major [out][in] with one f32 scale per output row. Per layer the
 * seven matrices are wq, wk, wv, wo, wg (gate), wu (up), wd (down). */
typedef struct {
  const float* tok_emb;            /* [vocab][dim] */
  const int8_t* const* w;          /* [n_layers * 7] */
  const float* const* w_scale;     /* [n_layers * 7] */
  const float* const* attn_norm;   /* [n_layers] -> [dim] */
  const float* const* ffn_norm;    /* [n_layers] -> [dim] */
  const float* final_norm;         /* [dim] */
  const int8_t* w_out;             /* [vocab][dim] */
  const float* w_out_scale;        /* [vocab] */
} orc_weights;

typedef struct orc_model orc_model;

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_CAPACITY -2
#define ORC_ERR_OOM -3

int orc_create(const orc_config* cfg, const orc_weights* w, int n_threads, orc_model** out);
void orc_destroy(orc_model* m);
/* Layer-major prefill of tokens[0..n) at positions start_pos.. in chunks of
 * `chunk`. Writes the last position's logits [vocab]; if `hidden` is not
 * NULL also the last position's residual stream [dim] before the final norm.
 * The K/V cache persists across calls. */
int orc_prefill(orc_model* m, const int32_t* tokens, int n, int start_pos, int chunk, float* logits,
                float* hidden);
/* One layer alone over rows x [n][dim] at positions start_pos .. start_pos+n-1
 * (as one chunk), in place; K/V rows of earlier positions come from the cache. */
int orc_layer(orc_model* m, int layer, float* x, int n, int start_pos);
/* Codes decided by another implementation at the four quantisation points
 * of a layer (0 attention input [dim], 1 attention output [n_heads*head_dim],
 * 2 FFN input [dim], 3 SwiGLU output [ffn]); rows have a pitch of kmax bytes.
 * The oracle fills in where its own decisions differed. */
typedef struct {
  const int8_t* codes[4];
  const float* scales[4];
  int kmax;
  int64_t mismatches[4];        /* codes that differ */
  int64_t scale_mismatches[4];  /* row scales that differ */
  float max_margin[4];          /* largest distance of a differing code's f32 value from a half-integer tie */
  int max_code_diff[4];         /* largest |difference| of differing codes */
  float max_scale_rel[4];       /* largest relative difference of differing row scales */
} orc_force;
int orc_layer_forced(orc_model* m, int layer, float* x, int n, int start_pos, orc_force* f);
/* Final RMSNorm + quantise + output projection of one residual row [dim]. */
int orc_final_logits(const orc_model* m, const float* x_row, float* logits);
/* Per-token reference: prefill of one token at `pos`. */
int orc_forward_one(orc_model* m, int32_t token, int pos, float* logits);
/* K (which = 0) or V (which = 1) cache of a layer: [max_seq][n_kv_heads][head_dim]. */
const float* orc_kv(const orc_model* m, int layer, int which);
void orc_kv_reset(orc_model* m);

/* ---- the steps, one by one ---- */
void orc_quantize_row(const float* y, int k, int8_t* q, float* a_scale);
void orc_quantize_rows(const float* y, int rows, int k, int8_t* q, float* a_scale);
int32_t orc_dot_i8(const int8_t* a, const int8_t* w, int k);
void orc_gemm_i8(const int8_t* a, const int8_t* w, int m, int n, int k, int32_t* acc, int n_threads);
float orc_dequant(int32_t acc, float w_scale, float a_scale);
void orc_rmsnorm_row(const float* x, const float* g, int d, float eps, float* y);
void orc_rmsnorm_rows(const float* x, const float* g, int rows, int d, float eps, float* y);
void orc_rope_head(float* v, int hd, int pos, float theta);
void orc_rope_rows(float* x, int rows, int n_heads, int hd, int start_pos, float theta);
float orc_silu_mul(float g, float u);
/* Causal attention of `rows` queries q[rows][n_heads][hd] at positions
 * start_pos + i over keys/values [0 .. start_pos + i] of K,V
 * [*][n_kv_heads][hd]; writes o[rows][n_heads][hd]. */
void orc_attention(const float* q, const float* K, const float* V, int rows, int start_pos, int n_heads,
                   int n_kv_heads, int hd, float* o, int n_threads);

#ifdef __cplusplus
}
#endif
#endif
