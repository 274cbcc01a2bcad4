/*
 * CPU oracle of layer-major batched int8 prefill -- TEST INFRASTRUCTURE ONLY.
 * Only tests, the smoke check and the bench's CPU-baseline leg use it; see
 * oracle.h for the sources and the precision rules. Built with
 * -ffp-contract=off and without fast-math so every f32 operation written
 * here is one IEEE-754 round-to-nearest operation.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* A row-split parallel-for. "Batched Prefill", section "The Solution":  */
/* threads split the work by weight rows, each thread owning a disjoint, */
/* contiguous slice that it reads once. Splitting never changes any      */
/* single result: every output element is computed by one thread alone.  */
/* ------------------------------------------------------------------ */
typedef void (*orc_range_fn)(void* ctx, int begin, int end);
typedef struct { orc_range_fn fn; void* ctx; int begin, end; } orc_slice;

static void* orc_slice_main(void* p) {
  orc_slice* s = (orc_slice*)p;
  s->fn(s->ctx, s->begin, s->end);
  return NULL;
}

static void orc_parallel_for(int n, int n_threads, orc_range_fn fn, void* ctx) {
  if (n <= 0) return;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 128) n_threads = 128;
  if (n_threads > n) n_threads = n;
  if (n_threads == 1) { fn(ctx, 0, n); return; }
  pthread_t th[128];
  int ok[128];
  orc_slice sl[128];
  int per = (n + n_threads - 1) / n_threads;
  for (int t = 0; t < n_threads; ++t) {
    sl[t].fn = fn; sl[t].ctx = ctx;
    sl[t].begin = t * per;
    sl[t].end = (t + 1) * per < n ? (t + 1) * per : n;
    ok[t] = 0;
    if (sl[t].begin >= sl[t].end) continue;
    if (pthread_create(&th[t], NULL, orc_slice_main, &sl[t]) == 0) ok[t] = 1;
    else fn(ctx, sl[t].begin, sl[t].end);
  }
  for (int t = 0; t < n_threads; ++t)
    if (ok[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* Per-token absmax int8 activation quantiser.                           */
/* "Batched Prefill", section "The Solution": activations are quantised  */
/* once per batch and the same int8 token columns serve every output     */
/* row. Symmetric per-token absmax, in f32 (the precision in which the   */
/* integer codes are decided on both sides):                              */
/*   amax = max_k |y_k|, a_scale = amax / 127, inv = 127 / amax,          */
/*   q_k = clamp(round-half-even(y_k * inv), -127, 127);                  */
/*   amax == 0 gives q = 0 and a_scale = 0.                               */
/* ------------------------------------------------------------------ */
void orc_quantize_row(const float* y, int k, int8_t* q, float* a_scale) {
  float amax = 0.0f;
  for (int i = 0; i < k; ++i) {
    float a = fabsf(y[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    memset(q, 0, (size_t)k);
    *a_scale = 0.0f;
    return;
  }
  float inv = 127.0f / amax;
  for (int i = 0; i < k; ++i) {
    float t = y[i] * inv;
    float r = nearbyintf(t); /* default rounding mode: ties to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
  *a_scale = amax / 127.0f;
}

void orc_quantize_rows(const float* y, int rows, int k, int8_t* q, float* a_scale) {
  for (int r = 0; r < rows; ++r) orc_quantize_row(y + (size_t)r * k, k, q + (size_t)r * k, a_scale + r);
}

/* ------------------------------------------------------------------ */
/* int8 x int8 -> int32 dot product and GEMM.                            */
/* "Batched Prefill", sections "The Solution" and "Correctness": one     */
/* weight row is dotted against many token columns; the sum is an exact  */
/* integer, so the batched GEMM equals the per-token GEMV bit for bit.   */
/* |acc| <= 127 * 127 * k < 2^31 for k <= 133,000.                       */
/* ------------------------------------------------------------------ */
int32_t orc_dot_i8(const int8_t* a, const int8_t* w, int k) {
  int32_t acc = 0;
  for (int i = 0; i < k; ++i) acc += (int32_t)a[i] * (int32_t)w[i];
  return acc;
}

typedef struct { const int8_t *a, *w; int m, n, k; int32_t* acc; } orc_gemm_ctx;

static void orc_gemm_rows(void* p, int r0, int r1) {
  orc_gemm_ctx* c = (orc_gemm_ctx*)p;
  for (int r = r0; r < r1; ++r) {
    const int8_t* wr = c->w + (size_t)r * c->k;
    for (int t = 0; t < c->m; ++t) c->acc[(size_t)t * c->n + r] = orc_dot_i8(c->a + (size_t)t * c->k, wr, c->k);
  }
}

/* acc[t][r] = sum_i a[t][i] * w[r][i]; a is [m][k] (tokens), w is [n][k] (rows). */
void orc_gemm_i8(const int8_t* a, const int8_t* w, int m, int n, int k, int32_t* acc, int n_threads) {
  orc_gemm_ctx c = {a, w, m, n, k, acc};
  orc_parallel_for(n, n_threads, orc_gemm_rows, &c);
}

/* Dequantising epilogue, f32 in the fixed order (float(acc) * w_scale) * a_scale. */
float orc_dequant(int32_t acc, float w_scale, float a_scale) {
  float f = (float)acc;
  f = f * w_scale;
  f = f * a_scale;
  return f;
}

/* ------------------------------------------------------------------ */
/* RMSNorm ("Single-pass prefill": the final RMSNorm before the output   */
/* projection; the same norm precedes attention and FFN in each block):  */
/*   y_k = x_k / sqrt(mean_j x_j^2 + eps) * g_k, in double.              */
/* ------------------------------------------------------------------ */
void orc_rmsnorm_row(const float* x, const float* g, int d, float eps, float* y) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += (double)x[i] * (double)x[i];
  double r = 1.0 / sqrt(ss / (double)d + (double)eps);
  for (int i = 0; i < d; ++i) y[i] = (float)((double)x[i] * r * (double)g[i]);
}

void orc_rmsnorm_rows(const float* x, const float* g, int rows, int d, float eps, float* y) {
  for (int r = 0; r < rows; ++r) orc_rmsnorm_row(x + (size_t)r * d, g, d, eps, y + (size_t)r * d);
}

/* ------------------------------------------------------------------ */
/* Rotary position embedding of one head at absolute position `pos`.     */
/* Pairs (j, j + hd/2) for j < hd/2 are rotated by pos * theta^(-2j/hd), */
/* in double.                                                            */
/* ------------------------------------------------------------------ */
void orc_rope_head(float* v, int hd, int pos, float theta) {
  int half = hd / 2;
  for (int j = 0; j < half; ++j) {
    double freq = pow((double)theta, -2.0 * (double)j / (double)hd);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double a = v[j], b = v[j + half];
    v[j] = (float)(a * c - b * s);
    v[j + half] = (float)(a * s + b * c);
  }
}

void orc_rope_rows(float* x, int rows, int n_heads, int hd, int start_pos, float theta) {
  for (int r = 0; r < rows; ++r)
    for (int h = 0; h < n_heads; ++h) orc_rope_head(x + ((size_t)r * n_heads + h) * hd, hd, start_pos + r, theta);
}

/* SwiGLU: silu(g) * u = g / (1 + exp(-g)) * u, in double. */
float orc_silu_mul(float g, float u) {
  double gd = (double)g;
  return (float)(gd / (1.0 + exp(-gd)) * (double)u);
}

/* ------------------------------------------------------------------ */
/* Causal attention. "Single-pass prefill": position i attends over the  */
/* K/V history kv[layer][0..i], already written because earlier          */
/* positions are processed first. Query head h reads KV head             */
/* h / (n_heads / n_kv_heads). In double:                                 */
/*   s_j = (q . k_j) / sqrt(hd), p_j = exp(s_j - max s),                  */
/*   o = sum_j p_j v_j / sum_j p_j.                                       */
/* ------------------------------------------------------------------ */
typedef struct {
  const float *q, *K, *V;
  int rows, start_pos, n_heads, n_kv_heads, hd;
  float* o;
} orc_attn_ctx;

static void orc_attn_items(void* p, int i0, int i1) {
  orc_attn_ctx* c = (orc_attn_ctx*)p;
  int group = c->n_heads / c->n_kv_heads;
  double scale = 1.0 / sqrt((double)c->hd);
  for (int it = i0; it < i1; ++it) {
    int i = it / c->n_heads, h = it % c->n_heads;
    int kvh = h / group;
    int n_keys = c->start_pos + i + 1;
    const float* qh = c->q + ((size_t)i * c->n_heads + h) * c->hd;
    double* s = (double*)malloc(sizeof(double) * (size_t)n_keys);
    double mx = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
      const float* kj = c->K + ((size_t)j * c->n_kv_heads + kvh) * c->hd;
      double d = 0.0;
      for (int e = 0; e < c->hd; ++e) d += (double)qh[e] * (double)kj[e];
      s[j] = d * scale;
      if (s[j] > mx) mx = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < n_keys; ++j) {
      s[j] = exp(s[j] - mx);
      l += s[j];
    }
    float* oh = c->o + ((size_t)i * c->n_heads + h) * c->hd;
    for (int e = 0; e < c->hd; ++e) {
      double acc = 0.0;
      for (int j = 0; j < n_keys; ++j) acc += s[j] * (double)c->V[((size_t)j * c->n_kv_heads + kvh) * c->hd + e];
      oh[e] = (float)(acc / l);
    }
    free(s);
  }
}

void orc_attention(const float* q, const float* K, const float* V, int rows, int start_pos, int n_heads,
                   int n_kv_heads, int hd, float* o, int n_threads) {
  orc_attn_ctx c = {q, K, V, rows, start_pos, n_heads, n_kv_heads, hd, o};
  orc_parallel_for(rows * n_heads, n_threads, orc_attn_items, &c);
}

/* ------------------------------------------------------------------ */
/* The model.                                                            */
/* ------------------------------------------------------------------ */
struct orc_model {
  orc_config cfg;
  orc_weights w;
  int n_threads;
  float* kcache; /* [n_layers][max_seq][n_kv_heads][head_dim] */
  float* vcache;
};

static size_t orc_kv_layer_elems(const orc_config* c) {
  return (size_t)c->max_seq * c->n_kv_heads * c->head_dim;
}

int orc_create(const orc_config* cfg, const orc_weights* w, int n_threads, orc_model** out) {
  if (!cfg || !w || !out) return ORC_ERR_ARG;
  if (cfg->dim <= 0 || cfg->n_layers <= 0 || cfg->n_heads <= 0 || cfg->n_kv_heads <= 0 || cfg->head_dim <= 0 ||
      (cfg->head_dim % 2) || cfg->ffn <= 0 || cfg->vocab <= 0 || cfg->max_seq <= 0 ||
      (cfg->n_heads % cfg->n_kv_heads))
    return ORC_ERR_ARG;
  orc_model* m = (orc_model*)calloc(1, sizeof *m);
  if (!m) return ORC_ERR_OOM;
  m->cfg = *cfg;
  m->w = *w;
  m->n_threads = n_threads < 1 ? 1 : n_threads;
  size_t n = orc_kv_layer_elems(cfg) * (size_t)cfg->n_layers;
  m->kcache = (float*)calloc(n, sizeof(float));
  m->vcache = (float*)calloc(n, sizeof(float));
  if (!m->kcache || !m->vcache) {
    orc_destroy(m);
    return ORC_ERR_OOM;
  }
  *out = m;
  return ORC_OK;
}

void orc_destroy(orc_model* m) {
  if (!m) return;
  free(m->kcache);
  free(m->vcache);
  free(m);
}

const float* orc_kv(const orc_model* m, int layer, int which) {
  if (!m || layer < 0 || layer >= m->cfg.n_layers) return NULL;
  return (which ? m->vcache : m->kcache) + orc_kv_layer_elems(&m->cfg) * (size_t)layer;
}

void orc_kv_reset(orc_model* m) {
  if (!m) return;
  size_t n = orc_kv_layer_elems(&m->cfg) * (size_t)m->cfg.n_layers;
  memset(m->kcache, 0, n * sizeof(float));
  memset(m->vcache, 0, n * sizeof(float));
}

/* out[t][r] = dequant(acc[t][r]) for an [rows][n] block. */
static void orc_dequant_block(const int32_t* acc, const float* w_scale, const float* a_scale, int rows, int n,
                              float* out) {
  for (int t = 0; t < rows; ++t)
    for (int r = 0; r < n; ++r) out[(size_t)t * n + r] = orc_dequant(acc[(size_t)t * n + r], w_scale[r], a_scale[t]);
}

/* Scratch for one chunk of up to `cm` positions. */
typedef struct {
  float *y, *as, *qf, *kf, *vf, *o, *hb, *proj;
  int8_t* qa;
  int32_t *acc, *acc2;
} orc_work;

static void orc_work_free(orc_work* w) {
  free(w->y); free(w->as); free(w->qf); free(w->kf); free(w->vf); free(w->o); free(w->hb); free(w->proj);
  free(w->qa); free(w->acc); free(w->acc2);
}

static int orc_work_alloc(const orc_config* c, int cm, orc_work* w) {
  const size_t QD = (size_t)c->n_heads * c->head_dim, KVD = (size_t)c->n_kv_heads * c->head_dim;
  size_t kmax = (size_t)c->dim;
  if (QD > kmax) kmax = QD;
  if ((size_t)c->ffn > kmax) kmax = (size_t)c->ffn;
  memset(w, 0, sizeof *w);
  w->y = (float*)malloc(sizeof(float) * cm * kmax);
  w->as = (float*)malloc(sizeof(float) * cm);
  w->qf = (float*)malloc(sizeof(float) * cm * QD);
  w->kf = (float*)malloc(sizeof(float) * cm * KVD);
  w->vf = (float*)malloc(sizeof(float) * cm * KVD);
  w->o = (float*)malloc(sizeof(float) * cm * QD);
  w->hb = (float*)malloc(sizeof(float) * cm * c->ffn);
  w->proj = (float*)malloc(sizeof(float) * cm * kmax);
  w->qa = (int8_t*)malloc((size_t)cm * kmax);
  w->acc = (int32_t*)malloc(sizeof(int32_t) * cm * kmax);
  w->acc2 = (int32_t*)malloc(sizeof(int32_t) * cm * c->ffn);
  if (!w->y || !w->as || !w->qf || !w->kf || !w->vf || !w->o || !w->hb || !w->proj || !w->qa || !w->acc ||
      !w->acc2) {
    orc_work_free(w);
    return ORC_ERR_OOM;
  }
  return ORC_OK;
}

/* Quantise rows as the method does; if `f` is given, compare the result with
 * the codes another implementation decided for the same quantisation point
 * and continue with those (see orc_layer_forced). */
static void orc_quantize_forced(const float* y, int rows, int k, int8_t* qa, float* as, orc_force* f, int pt,
                                int row0) {
  orc_quantize_rows(y, rows, k, qa, as);
  if (!f) return;
  for (int r = 0; r < rows; ++r) {
    const int8_t* fc = f->codes[pt] + (size_t)(row0 + r) * f->kmax;
    const float fs = f->scales[pt][row0 + r];
    if (fs != as[r]) {
      f->scale_mismatches[pt] += 1;
      float rel = fabsf(fs - as[r]) / (as[r] > 0.0f ? as[r] : 1.0f);
      if (rel > f->max_scale_rel[pt]) f->max_scale_rel[pt] = rel;
    }
    float amax_row = 0.0f;
    for (int i = 0; i < k; ++i) {
      float a = fabsf(y[(size_t)r * k + i]);
      if (a > amax_row) amax_row = a;
    }
    const float inv = amax_row == 0.0f ? 0.0f : 127.0f / amax_row;
    for (int i = 0; i < k; ++i) {
      const int8_t mine = qa[(size_t)r * k + i];
      if (mine != fc[i]) {
        f->mismatches[pt] += 1;
        int d = mine - fc[i];
        if (d < 0) d = -d;
        if (d > f->max_code_diff[pt]) f->max_code_diff[pt] = d;
        const float t = y[(size_t)r * k + i] * inv;
        const float margin = fabsf(t - (floorf(t) + 0.5f));
        if (margin > f->max_margin[pt]) f->max_margin[pt] = margin;
      }
      qa[(size_t)r * k + i] = fc[i];
    }
    as[r] = fs;
  }
}

/*
 * One decoder layer over one chunk of C positions pos0 .. pos0+C-1, in place
 * on the residual rows x [C][dim]. "Batched Prefill", "The Solution": the
 * chunk is quantised once per projection input and every output row reuses
 * it; "What Stays Sequential": attention runs per position, after the
 * chunk's K/V rows are written (each K/V row depends only on its own
 * position, so writing the chunk's rows first changes no position's history).
 */
static void orc_layer_chunk(orc_model* m, orc_work* w, int L, float* x, int C, int pos0, orc_force* f,
                            int row0) {
  const orc_config* c = &m->cfg;
  const int D = c->dim, H = c->n_heads, HKV = c->n_kv_heads, HD = c->head_dim, F = c->ffn;
  const int QD = H * HD, KVD = HKV * HD;
  const size_t kvl = orc_kv_layer_elems(c);
  const int8_t* const* W = m->w.w + 7 * L;
  const float* const* S = m->w.w_scale + 7 * L;
  float* Kc = m->kcache + kvl * L;
  float* Vc = m->vcache + kvl * L;

  /* attention block: norm -> quantise once -> Q, K, V projections */
  orc_rmsnorm_rows(x, m->w.attn_norm[L], C, D, c->rms_eps, w->y);
  orc_quantize_forced(w->y, C, D, w->qa, w->as, f, 0, row0);
  orc_gemm_i8(w->qa, W[0], C, QD, D, w->acc, m->n_threads);
  orc_dequant_block(w->acc, S[0], w->as, C, QD, w->qf);
  orc_gemm_i8(w->qa, W[1], C, KVD, D, w->acc, m->n_threads);
  orc_dequant_block(w->acc, S[1], w->as, C, KVD, w->kf);
  orc_gemm_i8(w->qa, W[2], C, KVD, D, w->acc, m->n_threads);
  orc_dequant_block(w->acc, S[2], w->as, C, KVD, w->vf);

  /* RoPE at absolute positions, then write the chunk's K/V rows */
  orc_rope_rows(w->qf, C, H, HD, pos0, c->rope_theta);
  orc_rope_rows(w->kf, C, HKV, HD, pos0, c->rope_theta);
  for (int i = 0; i < C; ++i) {
    memcpy(Kc + (size_t)(pos0 + i) * KVD, w->kf + (size_t)i * KVD, sizeof(float) * KVD);
    memcpy(Vc + (size_t)(pos0 + i) * KVD, w->vf + (size_t)i * KVD, sizeof(float) * KVD);
  }

  /* causal attention per position over kv[0 .. pos] */
  orc_attention(w->qf, Kc, Vc, C, pos0, H, HKV, HD, w->o, m->n_threads);

  /* O projection + residual */
  orc_quantize_forced(w->o, C, QD, w->qa, w->as, f, 1, row0);
  orc_gemm_i8(w->qa, W[3], C, D, QD, w->acc, m->n_threads);
  orc_dequant_block(w->acc, S[3], w->as, C, D, w->proj);
  for (size_t e = 0; e < (size_t)C * D; ++e) x[e] = x[e] + w->proj[e];

  /* FFN: norm -> quantise -> gate, up -> SwiGLU -> quantise -> down + residual */
  orc_rmsnorm_rows(x, m->w.ffn_norm[L], C, D, c->rms_eps, w->y);
  orc_quantize_forced(w->y, C, D, w->qa, w->as, f, 2, row0);
  orc_gemm_i8(w->qa, W[4], C, F, D, w->acc, m->n_threads);
  orc_gemm_i8(w->qa, W[5], C, F, D, w->acc2, m->n_threads);
  for (int i = 0; i < C; ++i)
    for (int j = 0; j < F; ++j) {
      size_t e = (size_t)i * F + j;
      float g = orc_dequant(w->acc[e], S[4][j], w->as[i]);
      float u = orc_dequant(w->acc2[e], S[5][j], w->as[i]);
      w->hb[e] = orc_silu_mul(g, u);
    }
  orc_quantize_forced(w->hb, C, F, w->qa, w->as, f, 3, row0);
  orc_gemm_i8(w->qa, W[6], C, D, F, w->acc, m->n_threads);
  orc_dequant_block(w->acc, S[6], w->as, C, D, w->proj);
  for (size_t e = 0; e < (size_t)C * D; ++e) x[e] = x[e] + w->proj[e];
}

/* "Single-pass prefill": final RMSNorm + output projection of one row. */
int orc_final_logits(const orc_model* m, const float* x_row, float* logits) {
  if (!m || !x_row || !logits) return ORC_ERR_ARG;
  const orc_config* c = &m->cfg;
  float* y = (float*)malloc(sizeof(float) * c->dim);
  int8_t* q = (int8_t*)malloc((size_t)c->dim);
  int32_t* acc = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->vocab);
  if (!y || !q || !acc) {
    free(y); free(q); free(acc);
    return ORC_ERR_OOM;
  }
  float as;
  orc_rmsnorm_row(x_row, m->w.final_norm, c->dim, c->rms_eps, y);
  orc_quantize_row(y, c->dim, q, &as);
  orc_gemm_i8(q, m->w.w_out, 1, c->vocab, c->dim, acc, m->n_threads);
  for (int v = 0; v < c->vocab; ++v) logits[v] = orc_dequant(acc[v], m->w.w_out_scale[v], as);
  free(y); free(q); free(acc);
  return ORC_OK;
}

/* Layer L alone over rows x [n][dim] at positions start_pos .. (one chunk),
 * in place; K/V rows of positions < start_pos come from the cache. */
int orc_layer(orc_model* m, int layer, float* x, int n, int start_pos) {
  if (!m || !x || n <= 0 || start_pos < 0 || layer < 0 || layer >= m->cfg.n_layers) return ORC_ERR_ARG;
  if ((int64_t)start_pos + n > m->cfg.max_seq) return ORC_ERR_CAPACITY;
  orc_work w;
  if (orc_work_alloc(&m->cfg, n, &w) != ORC_OK) return ORC_ERR_OOM;
  orc_layer_chunk(m, &w, layer, x, n, start_pos, NULL, 0);
  orc_work_free(&w);
  return ORC_OK;
}

/* Layer L over rows x [n][dim] (one chunk at start_pos), taking at each of
 * its four quantisation points (0 attention input, 1 attention output,
 * 2 FFN input, 3 SwiGLU output) the codes and scales of `f` in place of its
 * own, after recording where its own decision differs. */
int orc_layer_forced(orc_model* m, int layer, float* x, int n, int start_pos, orc_force* f) {
  if (!m || !x || !f || n <= 0 || start_pos < 0 || layer < 0 || layer >= m->cfg.n_layers) return ORC_ERR_ARG;
  if ((int64_t)start_pos + n > m->cfg.max_seq) return ORC_ERR_CAPACITY;
  orc_work w;
  if (orc_work_alloc(&m->cfg, n, &w) != ORC_OK) return ORC_ERR_OOM;
  orc_layer_chunk(m, &w, layer, x, n, start_pos, f, 0);
  orc_work_free(&w);
  return ORC_OK;
}

/*
 * Layer-major prefill. "Single-pass prefill", section "The fix": for each
 * layer the weights are read once and every prompt position is swept
 * through it; "Batched Prefill", section "The Solution": positions are
 * processed in chunks (the weights are read once per chunk). Only the last
 * position's logits are produced.
 */
int orc_prefill(orc_model* m, const int32_t* tokens, int n, int start_pos, int chunk, float* logits,
                float* hidden) {
  if (!m || !tokens || !logits || n <= 0 || chunk <= 0 || start_pos < 0) return ORC_ERR_ARG;
  const orc_config* c = &m->cfg;
  if ((int64_t)start_pos + n > c->max_seq) return ORC_ERR_CAPACITY;
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->vocab) return ORC_ERR_ARG;

  const int D = c->dim;
  const int CM = chunk < n ? chunk : n;
  orc_work w;
  if (orc_work_alloc(c, CM, &w) != ORC_OK) return ORC_ERR_OOM;
  float* x = (float*)malloc(sizeof(float) * (size_t)CM * D);
  float* xlast = (float*)malloc(sizeof(float) * (size_t)D);
  int rc = ORC_OK;
  if (!x || !xlast) {
    rc = ORC_ERR_OOM;
    goto done;
  }
  for (int c0 = 0; c0 < n; c0 += chunk) {
    const int C = (n - c0) < chunk ? (n - c0) : chunk;
    for (int i = 0; i < C; ++i) memcpy(x + (size_t)i * D, m->w.tok_emb + (size_t)tokens[c0 + i] * D, sizeof(float) * D);
    for (int L = 0; L < c->n_layers; ++L) orc_layer_chunk(m, &w, L, x, C, start_pos + c0, NULL, 0);
    if (c0 + C == n) memcpy(xlast, x + (size_t)(C - 1) * D, sizeof(float) * D);
  }
  if (hidden) memcpy(hidden, xlast, sizeof(float) * D);
  rc = orc_final_logits(m, xlast, logits);
done:
  orc_work_free(&w);
  free(x);
  free(xlast);
  return rc;
}

/* Per-token path: the prefill of a single token ("Single-pass prefill":
 * the old loop of one forward() per prompt token). */
int orc_forward_one(orc_model* m, int32_t token, int pos, float* logits) {
  return orc_prefill(m, &token, 1, pos, 1, logits, NULL);
}
