// Host runtime behind the C ABI of include/pp.h: model load and repack, the
// layer-major prefill loop, the streamed-mode prefetch ring, statistics and
// the single-step entry points. Every step of the computation runs in this
// library's kernels; the host only validates, sequences and copies.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pp_internal.cuh"

using namespace pp;

namespace {

thread_local std::string g_err;

void set_err(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
}

#define PP_CUDA(call)                                                                           \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess) {                                                                    \
      set_err("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__);      \
      return e_ == cudaErrorMemoryAllocation ? PP_ERR_OOM : PP_ERR_CUDA;                        \
    }                                                                                           \
  } while (0)

#define PP_TRY(expr)         \
  do {                       \
    int rc_ = (expr);        \
    if (rc_ != PP_OK) return rc_; \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets of one layer's tensors in its packed block (identical on the
// host, in the resident device copy and in every ring slot).
struct LayerLayout {
  size_t wqkv, wo, wgu, wd, sqkv, so, sgu, sd, attn_norm, ffn_norm, bytes;
  size_t weight_bytes;  // int8 weights + f32 scales (what the GEMMs read)
};

LayerLayout make_layout(const pp_config& c) {
  const size_t D = c.dim, QD = (size_t)c.n_heads * c.head_dim, QKV = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim,
               F = c.ffn;
  LayerLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.wqkv = take(QKV * D);
  L.wo = take(D * QD);
  L.wgu = take(2 * F * D);
  L.wd = take(D * F);
  L.sqkv = take(QKV * 4);
  L.so = take(D * 4);
  L.sgu = take(2 * F * 4);
  L.sd = take(D * 4);
  L.attn_norm = take(D * 4);
  L.ffn_norm = take(D * 4);
  L.bytes = off;
  L.weight_bytes = (QKV * D + D * QD + 2 * F * D + D * F) + 4 * (QKV + D + 2 * F + D);
  return L;
}

// Repack layer `l` of the caller's weights into `dst` (host memory):
// wq|wk|wv rows fused into one QKV matrix, the rows of every q and k head in
// RoPE pair order (row 2j + e of the head is its row j + e * hd/2, so the two
// members of a rotated pair are adjacent output columns); gate and up rows
// interleaved in blocks of 16 (16 gate rows, then the same 16 up rows) so that
// one GEMM tile holds both operands of SwiGLU.
void pack_layer(const pp_config& c, const LayerLayout& lay, const pp_weights& w, int l, uint8_t* dst) {
  const size_t D = c.dim, hd = c.head_dim, F = c.ffn, half = hd / 2;
  const size_t qr = c.n_heads * hd, kr = c.n_kv_heads * hd;
  const int8_t* const* W = w.w + 7 * l;
  const float* const* S = w.w_scale + 7 * l;
  uint8_t* p = dst + lay.wqkv;
  float* s = reinterpret_cast<float*>(dst + lay.sqkv);
  auto pair_rows = [&](const int8_t* src, const float* ssrc, size_t heads, int8_t* out, float* sout) {
    for (size_t h = 0; h < heads; ++h)
      for (size_t r = 0; r < hd; ++r) {
        const size_t from = h * hd + (r >> 1) + (r & 1) * half;
        memcpy(out + (h * hd + r) * D, src + from * D, D);
        sout[h * hd + r] = ssrc[from];
      }
  };
  pair_rows(W[0], S[0], c.n_heads, reinterpret_cast<int8_t*>(p), s);
  pair_rows(W[1], S[1], c.n_kv_heads, reinterpret_cast<int8_t*>(p + qr * D), s + qr);
  memcpy(p + (qr + kr) * D, W[2], kr * D);
  memcpy(s + qr + kr, S[2], kr * 4);
  memcpy(dst + lay.wo, W[3], D * qr);
  memcpy(dst + lay.so, S[3], D * 4);
  const size_t B = kSwiGluBlock;
  int8_t* gu = reinterpret_cast<int8_t*>(dst + lay.wgu);
  float* sgu = reinterpret_cast<float*>(dst + lay.sgu);
  for (size_t b = 0; b < F / B; ++b) {
    memcpy(gu + (2 * b) * B * D, W[4] + b * B * D, B * D);
    memcpy(gu + (2 * b + 1) * B * D, W[5] + b * B * D, B * D);
    memcpy(sgu + 2 * b * B, S[4] + b * B, B * 4);
    memcpy(sgu + (2 * b + 1) * B, S[5] + b * B, B * 4);
  }
  memcpy(dst + lay.wd, W[6], D * F);
  memcpy(dst + lay.sd, S[6], D * 4);
  memcpy(dst + lay.attn_norm, w.attn_norm[l], D * 4);
  memcpy(dst + lay.ffn_norm, w.ffn_norm[l], D * 4);
}

struct LayerPtrs {
  const int8_t *wqkv, *wo, *wgu, *wd;
  const float *sqkv, *so, *sgu, *sd, *attn_norm, *ffn_norm;
};

LayerPtrs layer_ptrs(const LayerLayout& lay, const uint8_t* base) {
  LayerPtrs p;
  p.wqkv = reinterpret_cast<const int8_t*>(base + lay.wqkv);
  p.wo = reinterpret_cast<const int8_t*>(base + lay.wo);
  p.wgu = reinterpret_cast<const int8_t*>(base + lay.wgu);
  p.wd = reinterpret_cast<const int8_t*>(base + lay.wd);
  p.sqkv = reinterpret_cast<const float*>(base + lay.sqkv);
  p.so = reinterpret_cast<const float*>(base + lay.so);
  p.sgu = reinterpret_cast<const float*>(base + lay.sgu);
  p.sd = reinterpret_cast<const float*>(base + lay.sd);
  p.attn_norm = reinterpret_cast<const float*>(base + lay.attn_norm);
  p.ffn_norm = reinterpret_cast<const float*>(base + lay.ffn_norm);
  return p;
}

struct EventPair {
  cudaEvent_t a, b;
};

// Events of one profiled layer visit: compute (a..b) and, streamed, the copy (c..d).
struct LayerVisitEv {
  int layer;
  cudaEvent_t a, b, c, d;
};

}  // namespace

struct pp_model {
  pp_config cfg{};
  int device = 0;
  int engine = PP_GEMM_MMA;
  LayerLayout lay{};
  cudaStream_t stream = nullptr;       // compute stream (owned)
  cudaStream_t copy_stream = nullptr;  // streamed mode: layer copies
  cudaEvent_t done = nullptr;          // recorded on the caller's stream at the end of every prefill
  // weights
  uint8_t* d_layers = nullptr;  // resident: n_layers packed blocks
  uint8_t* h_layers = nullptr;  // streamed: pinned host packed blocks
  uint8_t* ring[2] = {nullptr, nullptr};
  cudaEvent_t ring_ready[2] = {nullptr, nullptr};
  cudaEvent_t ring_free[2] = {nullptr, nullptr};
  float* emb = nullptr;
  float* final_norm = nullptr;
  int8_t* w_out = nullptr;
  float* s_out = nullptr;
  float* rope = nullptr;
  float* kc = nullptr;
  float* vc = nullptr;
  size_t kv_layer_floats = 0;  // floats from one layer's K (or V) rows to the next layer's
  size_t alloc_bytes = 0;      // device bytes this model allocated (test cap, pp_debug_alloc_cap)
  int loader_fault = 0;        // pp_debug_loader_fault
  KvSpace kvs;                 // kv_grow: reserved range, mapped as positions are written
  // scratch
  float *x = nullptr, *qkv = nullptr, *qr = nullptr, *o = nullptr, *h = nullptr, *as = nullptr, *logits = nullptr;
  int8_t* a8 = nullptr;
  __half* a16 = nullptr;
  int32_t* tok = nullptr;
  int* status = nullptr;
  float* trace = nullptr;  // optional residual-stream trace [(n_layers+1)][trace_pos][dim]
  int8_t* trace_codes = nullptr;  // [n_layers][4][trace_pos][kmax]
  float* trace_scales = nullptr;  // [n_layers][4][trace_pos]
  int trace_pos = 0;
  // tcgen05 engine: tensor maps of every weight matrix (per layer, or per ring
  // slot in streamed mode: qkv, o, gate/up, down) and of the fp16 activation
  // buffer viewed with each GEMM's k (dim, n_heads*head_dim, ffn)
  // weight maps: per weight matrix, one per tile width of k_gemm_tc (kTcBn) and
  // one for k_gemm_tw (chunks of at most 128 rows)
  std::vector<CUtensorMap> wmap;
  // activation maps of the fp16 code buffer viewed with each GEMM's k (0 dim, 1
  // n_heads*head_dim, 2 ffn): k_gemm_tc's, and k_gemm_tw's per token tile (kTwNt)
  CUtensorMap amap[3]{};
  CUtensorMap amap_tw[3][3]{};
  TcWorkspace tcws;  // stream-K partial tiles and counters of the projection GEMMs
  float* attn_part = nullptr;  // per-key-range partial attention state of one chunk
  size_t attn_part_bytes = 0;
  // chunk overlap (pp_set_chunk_overlap): consecutive chunks rotate over up to
  // kOverlap streams (the compute stream and ostream[]), each with its own
  // scratch set (the fields above hold the active one, sets[] all of them);
  // chunk k waits for chunk k-1's K/V rows of a layer (qkv_ev) before its
  // attention at that layer
  struct Scratch {
    float *x, *qkv, *qr, *o, *h, *as;
    int8_t* a8;
    __half* a16;
    TcWorkspace tcws;
    float* attn_part;
    size_t attn_part_bytes;
    CUtensorMap amap[3];
    CUtensorMap amap_tw[3][3];
  };
  // Up to kOverlap chunks in flight, one stream and scratch set each; a call uses
  // min(kOverlap, its chunks). Measured on the 350M workload (24 chunks of 32):
  // 8 / 16 / 24 / 32 streams gave 10.4 / 8.6 / 6.9 / 6.9 ms per call.
  static constexpr int kOverlap = 32;
  bool overlap = false;
  bool gemm_wide = false;  // the current call overlaps chunks: widest GEMM tiles, no stream-K
  int sets_alloc = 1;      // scratch sets fully allocated (set 0 at load)
  int streams_ready = 1;   // overlap streams (set 0: the model's stream) with their K/V events
  int active_set = 0;
  Scratch sets[kOverlap]{};
  cudaStream_t ostream[kOverlap - 1] = {};
  std::vector<cudaEvent_t> qkv_ev[kOverlap];
  // stats and timing
  pp_stats stats{};
  std::vector<cudaEvent_t> ev_pool;
  std::vector<EventPair> prof_pending;                 // profiled kernel launches
  std::vector<EventPair> prefetch_pending;             // (copy_done, needed) per layer visit
  std::vector<int> prefetch_layer;                     // the layer of each prefetch_pending entry
  // per-layer profile (opt-in)
  bool layer_prof = false;
  std::vector<pp_layer_profile> lprof;
  std::vector<LayerVisitEv> lprof_pending;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> copy_ev;  // copy start/end of each visit of the current call
  std::vector<void*> allocations;
  // streams whose next kernel follows a wait on another stream's event (wait_event)
  std::vector<cudaStream_t> plain_next;
  // CUDA graphs of repeated calls (pp_set_graphs): one executable graph per call
  // shape and buffer set, with the statistics one execution adds
  struct GraphEntry {
    const int32_t* d_tok;
    float* d_logits;
    int n, start_pos, chunk, overlap, seg;
    cudaGraphExec_t exec;
    pp_stats delta;
    uint64_t last_use;
  };
  static constexpr int kGraphCache = 8;
  bool graphs = false;
  bool capturing = false;
  std::vector<GraphEntry> gcache;
  uint64_t gclock = 0;
};

namespace {

int ev_get(pp_model* m, cudaEvent_t* e) {
  if (!m->ev_pool.empty()) {
    *e = m->ev_pool.back();
    m->ev_pool.pop_back();
    return PP_OK;
  }
  PP_CUDA(cudaEventCreate(e));
  return PP_OK;
}

// Wait for everything the model has enqueued: its own streams and the last
// prefill on a caller's stream (the `done` event).
int sync_model(pp_model* m) {
  PP_CUDA(cudaStreamSynchronize(m->stream));
  if (m->copy_stream) PP_CUDA(cudaStreamSynchronize(m->copy_stream));
  for (auto s : m->ostream)
    if (s) PP_CUDA(cudaStreamSynchronize(s));
  if (m->done) PP_CUDA(cudaEventSynchronize(m->done));
  return PP_OK;
}

// Fold finished event pairs into the statistics (after sync_model).
int collect(pp_model* m) {
  for (auto& p : m->prof_pending) {
    float ms = 0.f;
    PP_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
    m->stats.prof_ms += ms;
    m->stats.prof_launches += 1;
    m->ev_pool.push_back(p.a);
    m->ev_pool.push_back(p.b);
  }
  m->prof_pending.clear();
  for (size_t i = 0; i < m->prefetch_pending.size(); ++i) {
    const EventPair& p = m->prefetch_pending[i];
    float ms = 0.f;  // time from the copy's completion to the moment compute needed it
    PP_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
    if (ms >= 0.f)
      m->stats.prefetch_hits += 1;
    else
      m->stats.prefetch_misses += 1;
    if (m->layer_prof && i < m->prefetch_layer.size() && ms < 0.f)
      m->lprof[m->prefetch_layer[i]].wait_ms += -ms;
    m->ev_pool.push_back(p.a);
    m->ev_pool.push_back(p.b);
  }
  m->prefetch_pending.clear();
  m->prefetch_layer.clear();
  for (auto& v : m->lprof_pending) {
    float ms = 0.f;
    PP_CUDA(cudaEventElapsedTime(&ms, v.a, v.b));
    pp_layer_profile& lp = m->lprof[v.layer];
    lp.compute_ms += ms;
    lp.visits += 1;
    m->ev_pool.push_back(v.a);
    m->ev_pool.push_back(v.b);
    if (v.c) {
      PP_CUDA(cudaEventElapsedTime(&ms, v.c, v.d));
      lp.io_ms += ms;
      m->ev_pool.push_back(v.c);
      m->ev_pool.push_back(v.d);
    }
  }
  m->lprof_pending.clear();
  return PP_OK;
}

// Make `st` wait for event `e` recorded on another stream. The next kernel
// launched on `st` is then launched plainly stream-ordered, without
// programmatic early start: every cross-stream dependency (a streamed layer's
// copy into its ring slot, earlier chunks' K/V rows, the previous call on
// another stream) holds by plain stream order, whatever a kernel reads before
// its griddepcontrol.wait (the GEMM producer's first weight loads).
int wait_event(pp_model* m, cudaStream_t st, cudaEvent_t e) {
  PP_CUDA(cudaStreamWaitEvent(st, e, 0));
  if (std::find(m->plain_next.begin(), m->plain_next.end(), st) == m->plain_next.end()) m->plain_next.push_back(st);
  return PP_OK;
}

// Launch one kernel through fn(pdl) on stream st, counting it and, when its
// class is profiled, bracketing it with CUDA events. pdl is false for the
// first kernel after a wait_event on st.
template <class F>
int launch(pp_model* m, int cls, cudaStream_t st, F&& fn) {
  const bool prof = m->cfg.profile_kernel == cls;
  auto it = std::find(m->plain_next.begin(), m->plain_next.end(), st);
  const bool pdl = it == m->plain_next.end();
  if (!pdl) m->plain_next.erase(it);
  EventPair p{};
  if (prof) {
    PP_TRY(ev_get(m, &p.a));
    PP_TRY(ev_get(m, &p.b));
    PP_CUDA(cudaEventRecord(p.a, st));
  }
  cudaError_t e = fn(pdl);
  if (e != cudaSuccess) {
    set_err("kernel launch (class %d) failed: %s", cls, cudaGetErrorString(e));
    return PP_ERR_CUDA;
  }
  m->stats.kernel_launches += 1;
  if (prof) {
    PP_CUDA(cudaEventRecord(p.b, st));
    m->prof_pending.push_back(p);
  }
  return PP_OK;
}

// Stream-K workspace the tcgen05 engine plans for an m x n x k GEMM (either kernel).
void gemm_workspace_need(int m, int n, int k, size_t* part, size_t* cnt) {
  if (m <= kTwMaxRows)
    tw_workspace_need(m, n, k, part, cnt);
  else
    tc_workspace_need(m, n, k, part, cnt);
}

// K-extent of one exact f32 segment of the tcgen05 engine (pp_set_exact_segment).
std::atomic<int> g_tc_seg{kTcSegK};
int tc_segment() { return g_tc_seg.load(); }

// One projection GEMM of the layer whose weight block sits at map group `mg`
// (matrix `which`: 0 qkv, 1 o, 2 gate/up, 3 down).
int gemm(pp_model* m, cudaStream_t st, int epi, int mg, int which, const float* ws, const int8_t* w, int M, int N,
         int K, float* out, int ldo, const TcRope& rope = TcRope{}) {
  if (m->engine == PP_GEMM_TC) {
    const int kind = K == m->cfg.dim ? 0 : (K == m->cfg.ffn ? 2 : 1);
    const CUtensorMap* wm = &m->wmap[((size_t)mg * 4 + which) * 4];
    if (M <= kTwMaxRows) {  // short chunk: weights on the MMA's M side (k_gemm_tw)
      const int ti = tw_nt_index(M);
      m->stats.gemm_launches[epi][3 + ti] += 1;
      return launch(m, PP_KERNEL_GEMM, st, [&](bool pdl) {
        return launch_gemm_tw(epi, m->amap_tw[kind][ti], wm[3], kTwNt[ti], ws, m->as, M, N, K, out, ldo, nullptr,
                              tc_segment(), m->status, m->tcws, st, TcWaits{}, rope, m->gemm_wide, pdl,
                              /*early_w=*/true);
      });
    }
    const int bi = tc_bn_index(M, N, K, m->gemm_wide);
    m->stats.gemm_launches[epi][bi] += 1;
    return launch(m, PP_KERNEL_GEMM, st, [&](bool pdl) {
      return launch_gemm_tc(epi, m->amap[kind], wm[bi], kTcBn[bi], ws, m->as, M, N, K, out, ldo, nullptr, tc_segment(),
                            m->status, m->tcws, st, TcWaits{}, rope, m->gemm_wide, pdl, /*early_w=*/true);
    });
  }
  return launch(m, PP_KERNEL_GEMM, st, [&](bool) {  // plain launches
    return launch_gemm_mma(epi, m->a8, w, ws, m->as, M, N, K, out, ldo, nullptr, st);
  });
}

int make_weight_maps(pp_model* m, const uint8_t* block) {
  const pp_config& c = m->cfg;
  const LayerPtrs L = layer_ptrs(m->lay, block);
  const int D = c.dim, QD = c.n_heads * c.head_dim, QKV = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim, F = c.ffn;
  const int8_t* w[4] = {L.wqkv, L.wo, L.wgu, L.wd};
  const int n[4] = {QKV, D, 2 * F, D}, k[4] = {D, QD, D, F};
  // per matrix: one map per k_gemm_tc tile width (the width a launch uses depends on its
  // chunk's row count), then k_gemm_tw's
  for (int i = 0; i < 4; ++i) {
    for (int b = 0; b < 3; ++b) {
      CUtensorMap t;
      PP_CUDA(make_tmap_w(&t, w[i], n[i], k[i], kTcBn[b]));
      m->wmap.push_back(t);
    }
    CUtensorMap t;
    PP_CUDA(make_tmap_tw_weights(&t, w[i], n[i], k[i]));
    m->wmap.push_back(t);
  }
  return PP_OK;
}

std::atomic<long long> g_alloc_cap{0};

template <class T>
int dalloc(pp_model* m, T** p, size_t n) {
  const size_t bytes = std::max<size_t>(n * sizeof(T), 256);
  const long long cap = g_alloc_cap.load();
  if (cap > 0 && (long long)(m->alloc_bytes + bytes) > cap) {
    set_err("device allocation of %zu bytes would pass the test cap of %lld bytes", bytes, cap);
    return PP_ERR_OOM;
  }
  m->alloc_bytes += bytes;
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, std::max<size_t>(n * sizeof(T), 256));
  if (e != cudaSuccess) {
    set_err("cudaMalloc(%zu) failed: %s", n * sizeof(T), cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? PP_ERR_OOM : PP_ERR_CUDA;
  }
  m->allocations.push_back(v);
  *p = static_cast<T*>(v);
  return PP_OK;
}

int validate_cfg(const pp_config* c) {
  if (!c) return PP_ERR_ARG;
  const bool ok = c->dim > 0 && c->dim % 64 == 0 && c->n_layers > 0 && c->n_heads > 0 && c->n_kv_heads > 0 &&
                  c->n_heads % c->n_kv_heads == 0 && (c->head_dim == 64 || c->head_dim == 128) &&
                  64 % (c->n_heads / c->n_kv_heads) == 0 && (c->n_heads * c->head_dim) % 64 == 0 && c->ffn > 0 &&
                  c->ffn % 64 == 0 && c->vocab > 0 && c->max_seq > 0 && c->max_chunk > 0 &&
                  (c->mode == PP_MODE_RESIDENT || c->mode == PP_MODE_STREAMED) &&
                  (c->mode == PP_MODE_RESIDENT || c->ring_slots == 1 || c->ring_slots == 2) && c->rms_eps >= 0.f &&
                  c->rope_theta > 0.f && c->profile_kernel >= PP_KERNEL_NONE && c->profile_kernel < PP_KERNEL_COUNT &&
                  (c->loop_order == PP_LOOP_CHUNK_OUTER || c->loop_order == PP_LOOP_LAYER_OUTER);
  if (!ok) {
    set_err("invalid pp_config (dim%%64, head_dim in {64,128}, 64 %% (H/Hkv), ffn%%64, sizes > 0, mode, ring_slots, "
            "loop_order)");
    return PP_ERR_ARG;
  }
  return PP_OK;
}

// One scratch set (residual rows, activations, codes, attention and stream-K
// workspaces, the activation tensor maps) into the model's scratch fields.
// own_residual: the set holds the residual rows of every position of a call
// (layer-outer order); the extra sets of chunk overlap use set 0's for that.
int alloc_scratch(pp_model* m, bool own_residual = true) {
  const pp_config& c = m->cfg;
  const size_t D = c.dim, QD = (size_t)c.n_heads * c.head_dim,
               QKV = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim, F = c.ffn, MC = c.max_chunk;
  const size_t KMAX = std::max(std::max(D, QD), F);
  // residual stream: max_chunk rows chunk-outer, every position of a call layer-outer
  const bool all_rows = own_residual && c.loop_order == PP_LOOP_LAYER_OUTER;
  PP_TRY(dalloc(m, &m->x, (all_rows ? std::max(MC, (size_t)c.max_seq) : MC) * D));
  // QKV rows staged for the RoPE kernel (the tcgen05 path rotates in its QKV epilogue instead)
  if (m->engine != PP_GEMM_TC) PP_TRY(dalloc(m, &m->qkv, MC * QKV));
  PP_TRY(dalloc(m, &m->qr, MC * QD));
  PP_TRY(dalloc(m, &m->o, MC * QD));
  {
    // largest chunk at the end of the cache: the most tiles times the most key ranges
    const int rows = (int)std::min<size_t>(MC, (size_t)c.max_seq);
    m->attn_part_bytes = attention_workspace_bytes(rows, c.max_seq - rows, c.n_heads, c.n_kv_heads, c.head_dim);
    if (m->attn_part_bytes) PP_TRY(dalloc(m, &m->attn_part, m->attn_part_bytes / sizeof(float)));
  }
  PP_TRY(dalloc(m, &m->h, MC * F));
  PP_TRY(dalloc(m, &m->a8, MC * KMAX));
  PP_TRY(dalloc(m, &m->a16, MC * KMAX));
  PP_TRY(dalloc(m, &m->as, MC));
  PP_CUDA(cudaMemsetAsync(m->a16, 0, MC * KMAX * sizeof(__half), m->stream));
  if (m->engine == PP_GEMM_TC) {
    // stream-K workspace: the largest need over every chunk-row count and projection
    size_t part = 0, cnt = 0;
    const int shapes[4][2] = {{(int)QKV, (int)D}, {(int)D, (int)QD}, {(int)(2 * F), (int)D}, {(int)D, (int)F}};
    std::vector<size_t> row_counts = {32, 64, 128};  // the short-chunk kernel's token tiles
    for (size_t rows = 256; rows < MC + 256; rows += 256) row_counts.push_back(rows);
    for (size_t rows : row_counts)
      for (auto& sh : shapes) {
        size_t pb = 0, cc = 0;
        gemm_workspace_need((int)std::min(rows, MC), sh[0], sh[1], &pb, &cc);
        part = std::max(part, pb);
        cnt = std::max(cnt, cc);
      }
    if (part) {
      PP_TRY(dalloc(m, &m->tcws.part, part / sizeof(int32_t)));
      PP_TRY(dalloc(m, &m->tcws.cnt, cnt));
      PP_CUDA(cudaMemsetAsync(m->tcws.cnt, 0, cnt * sizeof(int), m->stream));
      m->tcws.part_bytes = part;
      m->tcws.counters = cnt;
    }
    const int ks[3] = {(int)D, (int)QD, (int)F};
    for (int i = 0; i < 3; ++i) {
      PP_CUDA(make_tmap_a(&m->amap[i], m->a16, (int)MC, ks[i]));
      for (int j = 0; j < 3; ++j) PP_CUDA(make_tmap_tw_tokens(&m->amap_tw[i][j], m->a16, (int)MC, ks[i], kTwNt[j]));
    }
  }
  return PP_OK;
}

// Make scratch set j the model's fields (the active set's pointers are kept in sets[]).
void use_scratch(pp_model* m, int j) {
  if (j == m->active_set) return;
  pp_model::Scratch& cur = m->sets[m->active_set];
  cur.x = m->x;
  cur.qkv = m->qkv;
  cur.qr = m->qr;
  cur.o = m->o;
  cur.h = m->h;
  cur.as = m->as;
  cur.a8 = m->a8;
  cur.a16 = m->a16;
  cur.tcws = m->tcws;
  cur.attn_part = m->attn_part;
  cur.attn_part_bytes = m->attn_part_bytes;
  memcpy(cur.amap, m->amap, sizeof m->amap);
  memcpy(cur.amap_tw, m->amap_tw, sizeof m->amap_tw);
  const pp_model::Scratch& o = m->sets[j];
  m->x = o.x;
  m->qkv = o.qkv;
  m->qr = o.qr;
  m->o = o.o;
  m->h = o.h;
  m->as = o.as;
  m->a8 = o.a8;
  m->a16 = o.a16;
  m->tcws = o.tcws;
  m->attn_part = o.attn_part;
  m->attn_part_bytes = o.attn_part_bytes;
  memcpy(m->amap, o.amap, sizeof m->amap);
  memcpy(m->amap_tw, o.amap_tw, sizeof m->amap_tw);
  m->active_set = j;
}

int load_impl(pp_model* m, const pp_weights* w) {
  const pp_config& c = m->cfg;
  PP_CUDA(cudaGetDevice(&m->device));
  // the tcgen05 engine tiles weight rows in multiples of 128
  const int qkv_rows = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  const bool tc_shapes = qkv_rows % 128 == 0 && c.dim % 128 == 0 && (2 * c.ffn) % 128 == 0;
  const bool tc = tc_available() && tc_shapes;
  if (c.gemm_engine == PP_GEMM_TC && !tc) {
    set_err(tc_shapes ? "the tcgen05 engine needs an sm_103 device"
                      : "the tcgen05 engine needs (H + 2 Hkv) hd, dim and 2 ffn to be multiples of 128");
    return PP_ERR_UNSUPPORTED;
  }
  if (c.gemm_engine != PP_GEMM_AUTO && c.gemm_engine != PP_GEMM_MMA && c.gemm_engine != PP_GEMM_TC) {
    set_err("unknown gemm_engine %d", c.gemm_engine);
    return PP_ERR_ARG;
  }
  m->engine = c.gemm_engine == PP_GEMM_MMA ? PP_GEMM_MMA : (tc ? PP_GEMM_TC : PP_GEMM_MMA);
  PP_CUDA(cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking));
  PP_CUDA(cudaEventCreateWithFlags(&m->done, cudaEventDisableTiming));
  m->lay = make_layout(c);
  const size_t D = c.dim, V = c.vocab;
  const size_t KVE = (size_t)c.n_layers * c.max_seq * c.n_kv_heads * c.head_dim;

  // global tensors
  PP_TRY(dalloc(m, &m->emb, V * D));
  PP_TRY(dalloc(m, &m->final_norm, D));
  PP_TRY(dalloc(m, &m->w_out, V * D));
  PP_TRY(dalloc(m, &m->s_out, V));
  PP_TRY(dalloc(m, &m->rope, (size_t)c.max_seq * c.head_dim));
  const size_t kv_row = (size_t)c.n_kv_heads * c.head_dim;  // floats per position per layer
  if (c.kv_grow) {
    // K regions 0..L-1 then V regions L..2L-1, each padded to the mapping granularity
    cudaError_t e = kv_space_reserve(&m->kvs, m->device, 2 * c.n_layers, (size_t)c.max_seq * kv_row * sizeof(float));
    if (e != cudaSuccess) {
      set_err("reserving the K/V address range failed: %s", cudaGetErrorString(e));
      return e == cudaErrorMemoryAllocation ? PP_ERR_OOM : PP_ERR_UNSUPPORTED;
    }
    m->kv_layer_floats = m->kvs.region_bytes / sizeof(float);
    m->kc = reinterpret_cast<float*>(m->kvs.base);
    m->vc = m->kc + (size_t)c.n_layers * m->kv_layer_floats;
  } else {
    PP_TRY(dalloc(m, &m->kc, KVE));
    PP_TRY(dalloc(m, &m->vc, KVE));
    m->kv_layer_floats = (size_t)c.max_seq * kv_row;
  }
  PP_CUDA(cudaMemcpy(m->emb, w->tok_emb, V * D * 4, cudaMemcpyHostToDevice));
  PP_CUDA(cudaMemcpy(m->final_norm, w->final_norm, D * 4, cudaMemcpyHostToDevice));
  PP_CUDA(cudaMemcpy(m->w_out, w->w_out, V * D, cudaMemcpyHostToDevice));
  PP_CUDA(cudaMemcpy(m->s_out, w->w_out_scale, V * 4, cudaMemcpyHostToDevice));
  if (!c.kv_grow) {
    PP_CUDA(cudaMemsetAsync(m->kc, 0, KVE * 4, m->stream));
    PP_CUDA(cudaMemsetAsync(m->vc, 0, KVE * 4, m->stream));
  }
  PP_CUDA(launch_rope_table(c.max_seq, c.head_dim, c.rope_theta, m->rope, m->stream));

  // scratch
  PP_TRY(alloc_scratch(m));
  PP_TRY(dalloc(m, &m->logits, V));
  PP_TRY(dalloc(m, &m->tok, (size_t)c.max_seq));
  PP_TRY(dalloc(m, &m->status, 1));
  PP_CUDA(cudaMemsetAsync(m->status, 0, sizeof(int), m->stream));

  // layers
  const size_t stride = m->lay.bytes;
  if (c.mode == PP_MODE_RESIDENT) {
    PP_TRY(dalloc(m, &m->d_layers, stride * c.n_layers));
    uint8_t* stage = nullptr;
    PP_CUDA(cudaMallocHost(&stage, stride));
    for (int l = 0; l < c.n_layers; ++l) {
      pack_layer(c, m->lay, *w, l, stage);
      cudaError_t e = cudaMemcpy(m->d_layers + stride * l, stage, stride, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        cudaFreeHost(stage);
        set_err("layer upload failed: %s", cudaGetErrorString(e));
        return PP_ERR_CUDA;
      }
    }
    cudaFreeHost(stage);
    if (m->engine == PP_GEMM_TC)
      for (int l = 0; l < c.n_layers; ++l) PP_TRY(make_weight_maps(m, m->d_layers + stride * l));
  } else {
    cudaError_t e = cudaHostAlloc(&m->h_layers, stride * c.n_layers, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      m->h_layers = nullptr;
      set_err("cudaHostAlloc(%zu) failed: %s", stride * c.n_layers, cudaGetErrorString(e));
      return PP_ERR_OOM;
    }
    for (int l = 0; l < c.n_layers; ++l) pack_layer(c, m->lay, *w, l, m->h_layers + stride * l);
    PP_CUDA(cudaStreamCreateWithFlags(&m->copy_stream, cudaStreamNonBlocking));
    for (int s = 0; s < c.ring_slots; ++s) {
      PP_TRY(dalloc(m, &m->ring[s], stride));
      PP_CUDA(cudaEventCreateWithFlags(&m->ring_ready[s], cudaEventDisableTiming));
      PP_CUDA(cudaEventCreateWithFlags(&m->ring_free[s], cudaEventDisableTiming));
      PP_CUDA(cudaEventRecord(m->ring_free[s], m->stream));
      if (m->engine == PP_GEMM_TC) PP_TRY(make_weight_maps(m, m->ring[s]));
    }
  }
  PP_CUDA(cudaStreamSynchronize(m->stream));
  return PP_OK;
}

void graphs_clear(pp_model* m);

void free_impl(pp_model* m) {
  if (m->stream) cudaStreamSynchronize(m->stream);
  if (m->copy_stream) cudaStreamSynchronize(m->copy_stream);
  for (auto s : m->ostream)
    if (s) cudaStreamSynchronize(s);
  if (m->done) {
    cudaEventSynchronize(m->done);
    cudaEventDestroy(m->done);
  }
  for (auto& p : m->prof_pending) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
  for (auto& p : m->prefetch_pending) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
  for (auto& v : m->lprof_pending) {
    cudaEventDestroy(v.a);
    cudaEventDestroy(v.b);
    if (v.c) { cudaEventDestroy(v.c); cudaEventDestroy(v.d); }
  }
  for (auto& e : m->copy_ev)
    if (e.first) { cudaEventDestroy(e.first); cudaEventDestroy(e.second); }
  for (auto e : m->ev_pool) cudaEventDestroy(e);
  graphs_clear(m);
  for (int s = 0; s < 2; ++s) {
    if (m->ring_ready[s]) cudaEventDestroy(m->ring_ready[s]);
    if (m->ring_free[s]) cudaEventDestroy(m->ring_free[s]);
  }
  for (int p = 0; p < pp_model::kOverlap; ++p)
    for (auto e : m->qkv_ev[p]) cudaEventDestroy(e);
  for (auto s : m->ostream)
    if (s) cudaStreamDestroy(s);
  for (void* p : m->allocations) cudaFree(p);
  if (m->kvs.base) kv_space_free(&m->kvs);
  if (m->h_layers) cudaFreeHost(m->h_layers);
  if (m->copy_stream) cudaStreamDestroy(m->copy_stream);
  if (m->stream) cudaStreamDestroy(m->stream);
  delete m;
}

int check_prefill_args(pp_model* m, int n, int start_pos, int chunk) {
  if (!m) { set_err("null model"); return PP_ERR_ARG; }
  if (n <= 0 || chunk <= 0 || start_pos < 0 || chunk > m->cfg.max_chunk) {
    set_err("bad prefill arguments: n=%d start_pos=%d chunk=%d (max_chunk %d)", n, start_pos, chunk, m->cfg.max_chunk);
    return PP_ERR_ARG;
  }
  if ((int64_t)start_pos + n > m->cfg.max_seq || (m->trace && (int64_t)start_pos + n > m->trace_pos)) {
    set_err("start_pos + n = %lld exceeds max_seq %d", (long long)start_pos + n, m->cfg.max_seq);
    return PP_ERR_CAPACITY;
  }
  return PP_OK;
}

// Streamed mode, before layer visit `v` of this call: make sure the copy of
// visit v is issued, issue the prefetch of visit v+1 into the other slot when
// the ring has two slots ("Predictive prefetch": the worker materialises block
// L+1 while block L computes), and make the compute stream wait for slot v.
int stream_layer(pp_model* m, cudaStream_t st, int v, int n_visits, const uint8_t** base) {
  const pp_config& c = m->cfg;
  const int S = c.ring_slots;
  const size_t stride = m->lay.bytes;
  auto issue_copy = [&](int visit) -> int {
    const int slot = visit % S;
    const int layer = visit % c.n_layers;
    PP_CUDA(cudaStreamWaitEvent(m->copy_stream, m->ring_free[slot], 0));
    cudaEvent_t c0 = nullptr, c1 = nullptr;
    if (m->layer_prof) {
      PP_TRY(ev_get(m, &c0));
      PP_TRY(ev_get(m, &c1));
      PP_CUDA(cudaEventRecord(c0, m->copy_stream));
    }
    PP_CUDA(cudaMemcpyAsync(m->ring[slot], m->h_layers + stride * layer, stride, cudaMemcpyHostToDevice,
                            m->copy_stream));
    if (m->layer_prof) {
      PP_CUDA(cudaEventRecord(c1, m->copy_stream));
      if ((int)m->copy_ev.size() <= visit) m->copy_ev.resize(visit + 1, {nullptr, nullptr});
      m->copy_ev[visit] = {c0, c1};
    }
    PP_CUDA(cudaEventRecord(m->ring_ready[slot], m->copy_stream));
    m->stats.h2d_bytes += (int64_t)stride;
    return PP_OK;
  };
  EventPair hp{};
  PP_TRY(ev_get(m, &hp.a));
  PP_TRY(ev_get(m, &hp.b));
  const bool prefetch = S == 2 && m->loader_fault == 0;
  if (v == 0 || !prefetch) PP_TRY(issue_copy(v));
  // The copy of visit v is now the newest work on the copy stream (with two
  // slots it was issued at visit v-1 and the copy of v+1 is issued below).
  PP_CUDA(cudaEventRecord(hp.a, m->copy_stream));  // copy of visit v done
  PP_CUDA(cudaEventRecord(hp.b, st));              // the compute stream reached layer v
  const int slot = v % S;
  PP_TRY(wait_event(m, st, m->ring_ready[slot]));
  if (prefetch && v + 1 < n_visits) PP_TRY(issue_copy(v + 1));
  m->prefetch_pending.push_back(hp);
  m->prefetch_layer.push_back(v % c.n_layers);
  *base = m->ring[slot];
  return PP_OK;
}

int trace_codes(pp_model* m, cudaStream_t cs, int layer, int point, int pos0, int C, int K) {
  if (!m->trace_codes) return PP_OK;
  const pp_config& c = m->cfg;
  const size_t kmax = std::max(std::max((size_t)c.dim, (size_t)c.n_heads * c.head_dim), (size_t)c.ffn);
  const size_t rec = (size_t)(layer * 4 + point) * m->trace_pos + pos0;
  PP_CUDA(cudaMemcpy2DAsync(m->trace_codes + rec * kmax, kmax, m->a8, K, K, C, cudaMemcpyDeviceToDevice, cs));
  if (m->trace_scales)
    PP_CUDA(cudaMemcpyAsync(m->trace_scales + rec, m->as, sizeof(float) * C, cudaMemcpyDeviceToDevice, cs));
  return PP_OK;
}

// One layer over the C rows of a chunk at positions pos0.. (residual rows x):
// attention block then FFN block, every projection an int8 GEMM over the chunk.
// kv_wait: the previous chunk's K/V event of the layer (chunk overlap),
// waited for before the attention reads the earlier rows; kv_done: recorded
// after this chunk's K/V rows of the layer are written and after that wait, so
// it stands for the K/V rows of this chunk and of every earlier chunk (a chunk
// two or three back runs on another stream and is covered only through it).
int layer_block(pp_model* m, cudaStream_t cs, int l, int mg, const uint8_t* base, float* x, int C, int pos0,
                cudaEvent_t kv_done = nullptr, cudaEvent_t kv_wait = nullptr) {
  const pp_config& c = m->cfg;
  const int D = c.dim, H = c.n_heads, Hkv = c.n_kv_heads, hd = c.head_dim, F = c.ffn;
  const int QD = H * hd, QKV = (H + 2 * Hkv) * hd;
  const size_t kvl = m->kv_layer_floats;
  __half* q16 = m->engine == PP_GEMM_TC ? m->a16 : nullptr;
  // the tcgen05 GEMMs read only the fp16 codes: the int8 copy is written for the
  // mma.sync engine and for the code trace
  int8_t* q8 = (m->engine == PP_GEMM_TC && !m->trace_codes) ? nullptr : m->a8;
  if (m->trace)
    PP_CUDA(cudaMemcpyAsync(m->trace + ((size_t)l * m->trace_pos + pos0) * D, x, sizeof(float) * C * D,
                            cudaMemcpyDeviceToDevice, cs));
  const LayerPtrs L = layer_ptrs(m->lay, base);
  float* kcl = m->kc + kvl * l;
  float* vcl = m->vc + kvl * l;
  // attention block
  PP_TRY(launch(m, PP_KERNEL_NORM_QUANT, cs, [&](bool pdl) {
    return launch_norm_quant(x, D, L.attn_norm, C, D, c.rms_eps, nullptr, q8, q16, m->as, cs, pdl);
  }));
  PP_TRY(trace_codes(m, cs, l, 0, pos0, C, D));
  if (m->engine == PP_GEMM_TC) {
    // QKV projection with RoPE and the K/V write in its epilogue
    TcRope rp;
    rp.table = m->rope;
    rp.pos0 = pos0;
    rp.H = H;
    rp.Hkv = Hkv;
    rp.hd = hd;
    rp.q_out = m->qr;
    rp.k_cache = kcl;
    rp.v_cache = vcl;
    PP_TRY(gemm(m, cs, EPI_ROPE, mg, 0, L.sqkv, L.wqkv, C, QKV, D, nullptr, QKV, rp));
  } else {
    PP_TRY(gemm(m, cs, EPI_STORE, mg, 0, L.sqkv, L.wqkv, C, QKV, D, m->qkv, QKV));
    PP_TRY(launch(m, PP_KERNEL_ROPE_KV, cs, [&](bool pdl) {
      return launch_rope_kv(m->qkv, C, pos0, H, Hkv, hd, m->rope, m->qr, kcl, vcl, cs, true, pdl);
    }));
  }
  if (kv_wait) PP_TRY(wait_event(m, cs, kv_wait));
  if (kv_done) PP_CUDA(cudaEventRecord(kv_done, cs));
  PP_TRY(launch(m, PP_KERNEL_ATTENTION, cs, [&](bool pdl) {
    return launch_attention(m->qr, kcl, vcl, C, pos0, H, Hkv, hd, m->o, m->attn_part, m->attn_part_bytes, cs, pdl);
  }));
  if (attention_workspace_bytes(C, pos0, H, Hkv, hd)) m->stats.kernel_launches += 1;  // the range merge
  PP_TRY(launch(m, PP_KERNEL_NORM_QUANT, cs, [&](bool pdl) {
    return launch_norm_quant(m->o, QD, nullptr, C, QD, 0.f, nullptr, q8, q16, m->as, cs, pdl);
  }));
  PP_TRY(trace_codes(m, cs, l, 1, pos0, C, QD));
  PP_TRY(gemm(m, cs, EPI_RESID, mg, 1, L.so, L.wo, C, D, QD, x, D));
  // FFN block
  PP_TRY(launch(m, PP_KERNEL_NORM_QUANT, cs, [&](bool pdl) {
    return launch_norm_quant(x, D, L.ffn_norm, C, D, c.rms_eps, nullptr, q8, q16, m->as, cs, pdl);
  }));
  PP_TRY(trace_codes(m, cs, l, 2, pos0, C, D));
  PP_TRY(gemm(m, cs, EPI_SWIGLU, mg, 2, L.sgu, L.wgu, C, 2 * F, D, m->h, F));
  PP_TRY(launch(m, PP_KERNEL_NORM_QUANT, cs, [&](bool pdl) {
    return launch_norm_quant(m->h, F, nullptr, C, F, 0.f, nullptr, q8, q16, m->as, cs, pdl);
  }));
  PP_TRY(trace_codes(m, cs, l, 3, pos0, C, F));
  PP_TRY(gemm(m, cs, EPI_RESID, mg, 3, L.sd, L.wd, C, D, F, x, D));
  return PP_OK;
}

// The weights of layer l for visit v: resident block, or (streamed) the ring
// slot its copy lands in, with the compute stream made to wait for that copy.
int layer_weights(pp_model* m, cudaStream_t cs, int l, int v, int n_visits, const uint8_t** base, int* mg) {
  if (m->cfg.mode == PP_MODE_STREAMED) {
    *mg = v % m->cfg.ring_slots;
    return stream_layer(m, cs, v, n_visits, base);
  }
  *mg = l;
  *base = m->d_layers + m->lay.bytes * l;
  return PP_OK;
}

// Final RMSNorm -> quantise -> output projection of the last position's row.
int head(pp_model* m, cudaStream_t cs, const float* xlast, float* d_logits) {
  const pp_config& c = m->cfg;
  const int D = c.dim;
  __half* q16 = m->engine == PP_GEMM_TC ? m->a16 : nullptr;
  PP_TRY(launch(m, PP_KERNEL_NORM_QUANT, cs, [&](bool pdl) {
    return launch_norm_quant(xlast, D, m->final_norm, 1, D, c.rms_eps, nullptr, m->a8, q16, m->as, cs, pdl);
  }));
  PP_TRY(launch(m, PP_KERNEL_LM_HEAD, cs, [&](bool pdl) {
    return launch_lm_head(m->a8, m->as, m->w_out, m->s_out, c.vocab, D, d_logits, cs, pdl);
  }));
  return PP_OK;
}

// Streams a call with chunk overlap uses: one per chunk, at most kOverlap.
int overlap_streams(int n, int chunk) { return std::min(pp_model::kOverlap, (n + chunk - 1) / chunk); }

// Scratch sets, streams and K/V events for `ns` chunks in flight. Runs before
// a call (never inside a graph capture). A step that fails leaves what it made
// in place (released with the model); a later call resumes from there.
int ensure_overlap(pp_model* m, int ns) {
  if (ns <= m->sets_alloc && ns <= m->streams_ready) return PP_OK;
  PP_TRY(sync_model(m));
  for (int j = m->sets_alloc; j < ns; ++j) {
    use_scratch(m, j);  // the set is (re)allocated into its fields
    const int rc = alloc_scratch(m, false);
    use_scratch(m, 0);
    if (rc != PP_OK) return rc;
    m->sets_alloc = j + 1;
  }
  for (int j = m->streams_ready; j < ns; ++j) {
    if (!m->ostream[j - 1]) PP_CUDA(cudaStreamCreateWithFlags(&m->ostream[j - 1], cudaStreamNonBlocking));
    m->streams_ready = j + 1;
  }
  for (int p = 0; p < ns; ++p)
    while ((int)m->qkv_ev[p].size() < m->cfg.n_layers) {
      cudaEvent_t e;
      PP_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
      m->qkv_ev[p].push_back(e);
    }
  PP_CUDA(cudaStreamSynchronize(m->stream));  // the new sets' initial clears
  return PP_OK;
}

int prefill_impl(pp_model* m, const int32_t* d_tok, int n, int start_pos, int chunk, float* d_logits,
                 cudaStream_t st) {
  const pp_config& c = m->cfg;
  const int D = c.dim;
  const bool streamed = c.mode == PP_MODE_STREAMED;
  const bool layer_outer = c.loop_order == PP_LOOP_LAYER_OUTER;
  const int n_chunks = (n + chunk - 1) / chunk;
  // streamed: one layer copy per (chunk, layer) chunk-outer, per layer layer-outer
  const int n_visits = layer_outer ? c.n_layers : n_chunks * c.n_layers;
  if (c.kv_grow) {
    // back the K/V rows this call writes (positions < start_pos + n) with device memory
    const size_t need = ((size_t)start_pos + n) * c.n_kv_heads * c.head_dim * sizeof(float);
    const long long cap = g_alloc_cap.load();
    const size_t grown = (need + m->kvs.gran - 1) / m->kvs.gran * m->kvs.gran * (size_t)m->kvs.n_regions;
    if (cap > 0 && grown > (size_t)m->kvs.mapped * m->kvs.n_regions &&
        (long long)(m->alloc_bytes + grown) > cap) {
      set_err("growing the K/V cache to %zu bytes would pass the test cap of %lld bytes", grown, cap);
      return PP_ERR_OOM;
    }
    cudaError_t e = kv_space_grow(&m->kvs, need);
    if (e != cudaSuccess) {
      set_err("growing the K/V cache to %lld positions failed: %s", (long long)start_pos + n, cudaGetErrorString(e));
      return e == cudaErrorMemoryAllocation ? PP_ERR_OOM : PP_ERR_CUDA;
    }
  }
  // The model's scratch, K/V cache and ring are shared by every call: order
  // this call after the previous one, whichever stream that one ran on.
  if (!m->capturing) PP_TRY(wait_event(m, st, m->done));  // a graph launch waits outside the graph
  if (streamed && st != m->stream) {
    // keep the ring's events on one compute stream
    cudaEvent_t e;
    PP_TRY(ev_get(m, &e));
    PP_CUDA(cudaEventRecord(e, st));
    PP_TRY(wait_event(m, m->stream, e));
    m->ev_pool.push_back(e);
  }
  cudaStream_t cs = streamed ? m->stream : st;
  // per-layer profile: events around every layer visit (compute) and its copy
  if (m->layer_prof) m->copy_ev.assign(n_visits, {nullptr, nullptr});
  auto visit_begin = [&](cudaEvent_t* a) -> int {
    *a = nullptr;
    if (!m->layer_prof) return PP_OK;
    PP_TRY(ev_get(m, a));
    PP_CUDA(cudaEventRecord(*a, cs));
    return PP_OK;
  };
  auto visit_end = [&](int l, int v, cudaEvent_t a) -> int {
    if (!m->layer_prof) return PP_OK;
    cudaEvent_t b;
    PP_TRY(ev_get(m, &b));
    PP_CUDA(cudaEventRecord(b, cs));
    LayerVisitEv e{l, a, b, nullptr, nullptr};
    if (streamed && v < (int)m->copy_ev.size()) {
      e.c = m->copy_ev[v].first;
      e.d = m->copy_ev[v].second;
      m->copy_ev[v] = {nullptr, nullptr};
    }
    m->lprof_pending.push_back(e);
    return PP_OK;
  };
  const bool overlap = m->overlap && !streamed && !layer_outer && !m->layer_prof && n > chunk;
  if (overlap) {
    // "Batched Prefill" with consecutive chunks on NS streams: chunk k runs on
    // stream k % NS with scratch set k % NS and waits, layer by layer, for the
    // K/V rows of every earlier chunk before its attention (chunk k-1's event,
    // recorded after chunk k-1's own wait, covers them all; a chunk's other
    // inputs are its own), so chunk k's layer l can fill the SMs the others
    // leave idle between their kernels. Chunk k-NS ran on the same stream: its
    // scratch set is free in stream order.
    const int NS = overlap_streams(n, chunk);
    if (NS > m->sets_alloc || NS > m->streams_ready) {
      set_err("chunk overlap needs %d scratch sets", NS);
      return PP_ERR_CUDA;
    }
    cudaStream_t S[pp_model::kOverlap];
    S[0] = cs;
    cudaEvent_t e;
    PP_TRY(ev_get(m, &e));
    PP_CUDA(cudaEventRecord(e, cs));
    for (int i = 1; i < NS; ++i) {
      S[i] = m->ostream[i - 1];
      PP_TRY(wait_event(m, S[i], e));
    }
    m->ev_pool.push_back(e);
    int rc = PP_OK, k = 0;
    // the other streams fill the CTA pairs a GEMM leaves idle: each GEMM takes the
    // least SM time (widest tile, no stream-K) rather than the least latency
    m->gemm_wide = true;
    for (int c0 = 0; c0 < n && rc == PP_OK; c0 += chunk, ++k) {
      const int p = k % NS, prev = (k + NS - 1) % NS;
      use_scratch(m, p);
      cudaStream_t sk = S[p];
      const int C = std::min(chunk, n - c0);
      const int pos0 = start_pos + c0;
      rc = launch(m, PP_KERNEL_EMBED, sk, [&](bool pdl) {
        return launch_embed(d_tok + c0, C, m->emb, c.vocab, D, m->x, m->status, sk, pdl);
      });
      for (int l = 0; l < c.n_layers && rc == PP_OK; ++l)
        rc = layer_block(m, sk, l, l, m->d_layers + m->lay.bytes * l, m->x, C, pos0, m->qkv_ev[p][l],
                         k > 0 ? m->qkv_ev[prev][l] : nullptr);
      if (rc == PP_OK && m->trace) {  // the chunk's rows leaving the last layer (disjoint per chunk)
        const cudaError_t e = cudaMemcpyAsync(m->trace + ((size_t)c.n_layers * m->trace_pos + pos0) * D, m->x,
                                              sizeof(float) * C * D, cudaMemcpyDeviceToDevice, sk);
        if (e != cudaSuccess) {
          set_err("trace copy failed: %s", cudaGetErrorString(e));
          rc = PP_ERR_CUDA;
        }
      }
      if (rc == PP_OK && c0 + C == n) rc = head(m, sk, m->x + (size_t)(C - 1) * D, d_logits);
    }
    use_scratch(m, 0);  // set 0 is the model's between calls
    m->gemm_wide = false;
    // the call ends on the caller's stream, also after an error: whatever the
    // other streams have queued is ordered before the caller's next work
    for (int i = 1; i < NS; ++i) {
      PP_TRY(ev_get(m, &e));
      PP_CUDA(cudaEventRecord(e, S[i]));
      PP_TRY(wait_event(m, cs, e));
      m->ev_pool.push_back(e);
    }
    PP_TRY(rc);
  } else if (!layer_outer) {
    // "Batched Prefill": for each chunk, every layer over the chunk's rows
    int visit = 0;
    for (int c0 = 0; c0 < n; c0 += chunk) {
      const int C = std::min(chunk, n - c0);
      const int pos0 = start_pos + c0;
      PP_TRY(launch(m, PP_KERNEL_EMBED, cs, [&](bool pdl) {
        return launch_embed(d_tok + c0, C, m->emb, c.vocab, D, m->x, m->status, cs, pdl);
      }));
      for (int l = 0; l < c.n_layers; ++l, ++visit) {
        const uint8_t* base;
        int mg;
        PP_TRY(layer_weights(m, cs, l, visit, n_visits, &base, &mg));
        cudaEvent_t ev;
        PP_TRY(visit_begin(&ev));
        PP_TRY(layer_block(m, cs, l, mg, base, m->x, C, pos0));
        PP_TRY(visit_end(l, visit, ev));
        if (streamed) PP_CUDA(cudaEventRecord(m->ring_free[visit % c.ring_slots], cs));
      }
      if (m->trace)
        PP_CUDA(cudaMemcpyAsync(m->trace + ((size_t)c.n_layers * m->trace_pos + pos0) * D, m->x,
                                sizeof(float) * C * D, cudaMemcpyDeviceToDevice, cs));
      if (c0 + C == n) PP_TRY(head(m, cs, m->x + (size_t)(C - 1) * D, d_logits));
    }
  } else {
    // "Single-pass prefill": for each layer, every chunk of the call; the
    // residual rows of all n positions stay in m->x between layers. With chunk
    // overlap the chunks of a layer rotate over the streams as in chunk-outer
    // order (their residual rows are disjoint slices of set 0's m->x); with
    // streamed weights every stream waits for the layer's copy and the ring
    // slot is freed only after every stream's work on the layer.
    const bool ovl = m->overlap && !m->layer_prof && n > chunk;
    const int NS = ovl ? overlap_streams(n, chunk) : 1;
    if (NS > m->sets_alloc || NS > m->streams_ready) {
      set_err("chunk overlap needs %d scratch sets", NS);
      return PP_ERR_CUDA;
    }
    cudaStream_t S[pp_model::kOverlap];
    S[0] = cs;
    for (int i = 1; i < NS; ++i) S[i] = ovl ? m->ostream[i - 1] : cs;
    auto fan = [&](bool out) -> int {  // out: the others wait for cs; in: cs waits for the others
      for (int i = 1; i < NS; ++i) {
        cudaEvent_t e;
        PP_TRY(ev_get(m, &e));
        PP_CUDA(cudaEventRecord(e, out ? cs : S[i]));
        PP_TRY(wait_event(m, out ? S[i] : cs, e));
        m->ev_pool.push_back(e);
      }
      return PP_OK;
    };
    PP_TRY(launch(m, PP_KERNEL_EMBED, cs, [&](bool pdl) {
      return launch_embed(d_tok, n, m->emb, c.vocab, D, m->x, m->status, cs, pdl);
    }));
    float* const x0 = m->x;
    if (ovl) {
      PP_TRY(fan(true));
      m->gemm_wide = true;
    }
    int rc = PP_OK;
    for (int l = 0; l < c.n_layers && rc == PP_OK; ++l) {
      const uint8_t* base;
      int mg;
      rc = layer_weights(m, cs, l, l, n_visits, &base, &mg);
      if (rc == PP_OK && ovl && streamed) rc = fan(true);
      cudaEvent_t ev = nullptr;
      if (rc == PP_OK) rc = visit_begin(&ev);
      int k = 0;
      for (int c0 = 0; c0 < n && rc == PP_OK; c0 += chunk, ++k) {
        const int p = ovl ? k % NS : 0;
        if (ovl) use_scratch(m, p);
        rc = layer_block(m, S[p], l, mg, base, x0 + (size_t)c0 * D, std::min(chunk, n - c0), start_pos + c0,
                         ovl ? m->qkv_ev[p][l] : nullptr, ovl && k > 0 ? m->qkv_ev[(k + NS - 1) % NS][l] : nullptr);
      }
      if (rc == PP_OK && ovl && streamed) rc = fan(false);
      if (rc == PP_OK) rc = visit_end(l, l, ev);
      if (rc == PP_OK && streamed) PP_CUDA(cudaEventRecord(m->ring_free[l % c.ring_slots], cs));
    }
    if (ovl) {
      use_scratch(m, 0);
      m->gemm_wide = false;
      const int rf = fan(false);  // also after an error (see chunk-outer order)
      if (rc == PP_OK) rc = rf;
    }
    PP_TRY(rc);
    if (m->trace)
      PP_CUDA(cudaMemcpyAsync(m->trace + ((size_t)c.n_layers * m->trace_pos + start_pos) * D, m->x,
                              sizeof(float) * n * D, cudaMemcpyDeviceToDevice, cs));
    PP_TRY(head(m, cs, x0 + (size_t)(n - 1) * D, d_logits));
  }
  if (streamed && st != m->stream) {
    cudaEvent_t e;
    PP_TRY(ev_get(m, &e));
    PP_CUDA(cudaEventRecord(e, m->stream));
    PP_TRY(wait_event(m, st, e));
    m->ev_pool.push_back(e);
  }
  if (!m->capturing) PP_CUDA(cudaEventRecord(m->done, st));
  m->stats.calls += 1;
  m->stats.chunks += n_chunks;
  m->stats.tokens += n;
  m->stats.weight_bytes_read += (int64_t)m->lay.weight_bytes * c.n_layers * n_chunks + (int64_t)c.vocab * D +
                                (int64_t)c.vocab * 4;
  return PP_OK;
}


// Statistics one graph execution adds (the counters its capture incremented).
pp_stats stats_delta(const pp_stats& a, const pp_stats& b) {
  pp_stats d = b;
  d.calls -= a.calls;
  d.chunks -= a.chunks;
  d.tokens -= a.tokens;
  d.weight_bytes_read -= a.weight_bytes_read;
  d.h2d_bytes -= a.h2d_bytes;
  d.prefetch_hits -= a.prefetch_hits;
  d.prefetch_misses -= a.prefetch_misses;
  d.kernel_launches -= a.kernel_launches;
  d.prof_launches -= a.prof_launches;
  d.prof_ms -= a.prof_ms;
  for (int e = 0; e < 5; ++e)
    for (int b2 = 0; b2 < 6; ++b2) d.gemm_launches[e][b2] -= a.gemm_launches[e][b2];
  return d;
}

void stats_add(pp_stats* s, const pp_stats& d) {
  s->calls += d.calls;
  s->chunks += d.chunks;
  s->tokens += d.tokens;
  s->weight_bytes_read += d.weight_bytes_read;
  s->h2d_bytes += d.h2d_bytes;
  s->kernel_launches += d.kernel_launches;
  for (int e = 0; e < 5; ++e)
    for (int b = 0; b < 6; ++b) s->gemm_launches[e][b] += d.gemm_launches[e][b];
}

void graphs_clear(pp_model* m) {
  for (auto& g : m->gcache) cudaGraphExecDestroy(g.exec);
  m->gcache.clear();
}

// One prefill call: through a cached CUDA graph of the whole call when graphs
// are on and the call qualifies (resident weights, no profiling, tracing or
// K/V growth), else launch by launch. A graph is captured from the model's own
// stream the first time a (buffers, n, start_pos, chunk) combination is seen
// and replayed on `st` afterwards; replay runs exactly the launches of the
// capture, so the results are the same bits.
int prefill_call(pp_model* m, const int32_t* d_tok, int n, int start_pos, int chunk, float* d_logits,
                 cudaStream_t st) {
  const pp_config& c = m->cfg;
  const bool layer_outer = c.loop_order == PP_LOOP_LAYER_OUTER;
  if (m->overlap && !m->layer_prof && n > chunk && (layer_outer || c.mode != PP_MODE_STREAMED))
    PP_TRY(ensure_overlap(m, overlap_streams(n, chunk)));
  const bool use_graph = m->graphs && c.mode == PP_MODE_RESIDENT && !c.kv_grow && c.profile_kernel == PP_KERNEL_NONE &&
                         !m->trace && !m->layer_prof;
  if (!use_graph) return prefill_impl(m, d_tok, n, start_pos, chunk, d_logits, st);
  const int ovl = m->overlap ? 1 : 0, seg = tc_segment();
  pp_model::GraphEntry* hit = nullptr;
  for (auto& g : m->gcache)
    if (g.d_tok == d_tok && g.d_logits == d_logits && g.n == n && g.start_pos == start_pos && g.chunk == chunk &&
        g.overlap == ovl && g.seg == seg)
      hit = &g;
  if (!hit) {
    if ((int)m->gcache.size() >= pp_model::kGraphCache) {  // drop the least recently used graph
      auto lru = std::min_element(m->gcache.begin(), m->gcache.end(),
                                  [](const pp_model::GraphEntry& a, const pp_model::GraphEntry& b) {
                                    return a.last_use < b.last_use;
                                  });
      PP_TRY(sync_model(m));  // its last replay may still run
      cudaGraphExecDestroy(lru->exec);
      m->gcache.erase(lru);
    }
    const pp_stats before = m->stats;
    const std::vector<cudaStream_t> plain = m->plain_next;
    m->plain_next.clear();
    PP_CUDA(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeRelaxed));
    m->capturing = true;
    const int rc = prefill_impl(m, d_tok, n, start_pos, chunk, d_logits, m->stream);
    m->capturing = false;
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(m->stream, &graph);
    const pp_stats after = m->stats;
    m->stats = before;  // nothing ran yet
    m->plain_next = plain;
    if (rc != PP_OK || ec != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      if (rc != PP_OK) return rc;
      set_err("capturing the prefill graph failed: %s", cudaGetErrorString(ec));
      return PP_ERR_CUDA;
    }
    pp_model::GraphEntry g{};
    g.d_tok = d_tok;
    g.d_logits = d_logits;
    g.n = n;
    g.start_pos = start_pos;
    g.chunk = chunk;
    g.overlap = ovl;
    g.seg = seg;
    g.delta = stats_delta(before, after);
    const cudaError_t ei = cudaGraphInstantiate(&g.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
      set_err("instantiating the prefill graph failed: %s", cudaGetErrorString(ei));
      return PP_ERR_CUDA;
    }
    m->gcache.push_back(g);
    hit = &m->gcache.back();
  }
  hit->last_use = ++m->gclock;
  // the model's scratch and K/V cache are shared with the previous call, whatever its stream
  PP_CUDA(cudaStreamWaitEvent(st, m->done, 0));
  PP_CUDA(cudaGraphLaunch(hit->exec, st));
  PP_CUDA(cudaEventRecord(m->done, st));
  stats_add(&m->stats, hit->delta);
  return PP_OK;
}
}  // namespace

// =====================================================================  C ABI
// ---------------------------------------------------------------- host-buffer checks
namespace {
// Device copies of one call's buffers, freed when the call returns.
class DeviceScratch {
 public:
  DeviceScratch() = default;
  DeviceScratch(const DeviceScratch&) = delete;
  DeviceScratch& operator=(const DeviceScratch&) = delete;
  ~DeviceScratch() {
    for (void* p : bufs_) cudaFree(p);
  }
  template <class T>
  int alloc(T** out, size_t n) {
    void* p = nullptr;
    const cudaError_t e = cudaMalloc(&p, std::max<size_t>(n * sizeof(T), 256));
    if (e != cudaSuccess) {
      set_err("cudaMalloc(%zu) failed: %s", n * sizeof(T), cudaGetErrorString(e));
      return e == cudaErrorMemoryAllocation ? PP_ERR_OOM : PP_ERR_CUDA;
    }
    bufs_.push_back(p);
    *out = static_cast<T*>(p);
    return PP_OK;
  }
  template <class T>
  int upload(T** out, const T* host, size_t n) {
    PP_TRY(alloc(out, n));
    PP_CUDA(cudaMemcpy(*out, host, n * sizeof(T), cudaMemcpyHostToDevice));
    return PP_OK;
  }

 private:
  std::vector<void*> bufs_;
};

// The GEMM of pp_debug_gemm_i8 (acc != NULL) or pp_debug_gemm_epilogue (out != NULL).
int debug_gemm(const int8_t* a, const int8_t* w, const float* w_scale, const float* a_scale, const float* resid,
               int32_t m, int32_t n, int32_t k, int32_t* acc, float* out) {
  if (!a || !w || m <= 0 || n <= 0 || k <= 0 || k % 64 || n % 32 || (out && (!w_scale || !a_scale))) {
    set_err("bad pp_debug_gemm arguments (k %% 64, n %% 32)");
    return PP_ERR_ARG;
  }
  const int32_t engine = n % 128 == 0 ? PP_GEMM_TC : PP_GEMM_MMA;
  const size_t mk = (size_t)m * k, mn = (size_t)m * n;
  DeviceScratch d;
  int8_t *da = nullptr, *dw = nullptr;
  __half* da16 = nullptr;
  PP_TRY(d.upload(&da, a, mk));
  PP_TRY(d.upload(&dw, w, (size_t)n * k));
  if (engine == PP_GEMM_TC) {
    PP_TRY(d.alloc(&da16, mk));
    PP_CUDA(launch_widen_i8(da, (long long)mk, da16, nullptr));
  }
  const uint16_t* a16 = reinterpret_cast<const uint16_t*>(da16);
  if (acc) {
    int32_t* dacc = nullptr;
    PP_TRY(d.alloc(&dacc, mn));
    PP_TRY(pp_op_gemm_acc(engine, da, a16, dw, m, n, k, dacc, nullptr));
    if (engine == PP_GEMM_TC) PP_TRY(pp_op_status(nullptr));
    PP_CUDA(cudaMemcpy(acc, dacc, mn * sizeof(int32_t), cudaMemcpyDeviceToHost));
    return PP_OK;
  }
  float *dws = nullptr, *das = nullptr, *dout = nullptr;
  PP_TRY(d.upload(&dws, w_scale, (size_t)n));
  PP_TRY(d.upload(&das, a_scale, (size_t)m));
  if (resid) {
    PP_TRY(d.upload(&dout, resid, mn));
  } else {
    PP_TRY(d.alloc(&dout, mn));
  }
  PP_TRY(pp_op_gemm(engine, resid ? PP_EPI_RESID : PP_EPI_STORE, da, a16, dw, dws, das, m, n, k, dout, n, nullptr));
  if (engine == PP_GEMM_TC) PP_TRY(pp_op_status(nullptr));
  PP_CUDA(cudaMemcpy(out, dout, mn * sizeof(float), cudaMemcpyDeviceToHost));
  return PP_OK;
}
}  // namespace

extern "C" {

const char* pp_status_str(int s) {
  switch (s) {
    case PP_OK: return "ok";
    case PP_ERR_ARG: return "invalid argument";
    case PP_ERR_CAPACITY: return "KV capacity exceeded";
    case PP_ERR_OOM: return "out of memory";
    case PP_ERR_CUDA: return "CUDA error";
    case PP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case PP_ERR_UNSUPPORTED: return "unsupported";
    default: return "unknown status";
  }
}

const char* pp_last_error(void) { return g_err.c_str(); }

int pp_model_load(const pp_config* cfg, const pp_weights* w, pp_model** out) {
  if (!out) { set_err("null out"); return PP_ERR_ARG; }
  *out = nullptr;
  PP_TRY(validate_cfg(cfg));
  if (!w || !w->tok_emb || !w->w || !w->w_scale || !w->attn_norm || !w->ffn_norm || !w->final_norm || !w->w_out ||
      !w->w_out_scale) {
    set_err("null weight pointer");
    return PP_ERR_ARG;
  }
  for (int i = 0; i < 7 * cfg->n_layers; ++i)
    if (!w->w[i] || !w->w_scale[i]) { set_err("null layer matrix %d", i); return PP_ERR_ARG; }
  for (int l = 0; l < cfg->n_layers; ++l)
    if (!w->attn_norm[l] || !w->ffn_norm[l]) { set_err("null norm gain %d", l); return PP_ERR_ARG; }
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess || ndev == 0) {
    set_err("no CUDA device: %s", cudaGetErrorString(e));
    return PP_ERR_CUDA;
  }
  pp_model* m = new pp_model();
  m->cfg = *cfg;
  int rc = load_impl(m, w);
  if (rc != PP_OK) {
    std::string keep = g_err;
    free_impl(m);
    g_err = keep;
    return rc;
  }
  *out = m;
  return PP_OK;
}

void pp_model_free(pp_model* m) {
  if (m) free_impl(m);
}

int pp_prefill_device(pp_model* m, const int32_t* d_tokens, int32_t n, int32_t start_pos, int32_t chunk,
                      float* d_logits, void* stream) {
  PP_TRY(check_prefill_args(m, n, start_pos, chunk));
  if (!d_tokens || !d_logits) { set_err("null device pointer"); return PP_ERR_ARG; }
  // NULL is the legacy default stream, as for every other entry point
  return prefill_call(m, d_tokens, n, start_pos, chunk, d_logits, static_cast<cudaStream_t>(stream));
}

int pp_prefill(pp_model* m, const int32_t* tokens, int32_t n, int32_t start_pos, int32_t chunk, float* logits_out) {
  PP_TRY(check_prefill_args(m, n, start_pos, chunk));
  if (!tokens || !logits_out) { set_err("null host pointer"); return PP_ERR_ARG; }
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= m->cfg.vocab) {
      set_err("token %d at index %d outside [0, %d)", tokens[i], i, m->cfg.vocab);
      return PP_ERR_ARG;
    }
  PP_CUDA(cudaMemcpyAsync(m->tok, tokens, sizeof(int32_t) * n, cudaMemcpyHostToDevice, m->stream));
  m->stats.h2d_bytes += (int64_t)sizeof(int32_t) * n;
  PP_TRY(prefill_call(m, m->tok, n, start_pos, chunk, m->logits, m->stream));
  PP_CUDA(cudaMemcpyAsync(logits_out, m->logits, sizeof(float) * m->cfg.vocab, cudaMemcpyDeviceToHost, m->stream));
  PP_CUDA(cudaStreamSynchronize(m->stream));
  PP_TRY(collect(m));
  return pp_device_status(m);
}

int pp_forward_one(pp_model* m, int32_t token, int32_t pos, float* logits_out) {
  return pp_prefill(m, &token, 1, pos, 1, logits_out);
}

int pp_device_status(pp_model* m) {
  if (!m) return PP_ERR_ARG;
  PP_TRY(sync_model(m));
  int s = 0;
  PP_CUDA(cudaMemcpy(&s, m->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (s != DEV_OK) PP_CUDA(cudaMemset(m->status, 0, sizeof(int)));
  if (s == DEV_BAD_TOKEN) { set_err("a token id outside [0, vocab) reached the device"); return PP_ERR_ARG; }
  if (s == DEV_TIMEOUT) {
    if (m->tcws.cnt) cudaMemset(m->tcws.cnt, 0, m->tcws.counters * sizeof(int));
    set_err("a bounded device wait gave up");
    return PP_ERR_DEVICE_TIMEOUT;
  }
  return PP_OK;
}

int pp_kv_reset(pp_model* m) {
  if (!m) return PP_ERR_ARG;
  const pp_config& c = m->cfg;
  const size_t KVE = (size_t)c.n_layers * c.max_seq * c.n_kv_heads * c.head_dim;
  PP_TRY(sync_model(m));
  if (c.kv_grow) {  // give the device memory back; the next call maps what it writes
    kv_space_release(&m->kvs);
    return PP_OK;
  }
  PP_CUDA(cudaMemsetAsync(m->kc, 0, KVE * 4, m->stream));
  PP_CUDA(cudaMemsetAsync(m->vc, 0, KVE * 4, m->stream));
  PP_CUDA(cudaStreamSynchronize(m->stream));
  return PP_OK;
}

int pp_kv_read(pp_model* m, int32_t layer, int32_t which, int32_t pos0, int32_t n_pos, float* out) {
  if (!m || !out || layer < 0 || layer >= m->cfg.n_layers || (which != 0 && which != 1) || pos0 < 0 || n_pos <= 0 ||
      (int64_t)pos0 + n_pos > m->cfg.max_seq) {
    set_err("bad pp_kv_read arguments");
    return PP_ERR_ARG;
  }
  const pp_config& c = m->cfg;
  const size_t row = (size_t)c.n_kv_heads * c.head_dim;
  if (c.kv_grow && ((size_t)pos0 + n_pos) * row * sizeof(float) > m->kvs.mapped) {
    set_err("pp_kv_read: positions [%d, %d) were never written since the last reset", pos0, pos0 + n_pos);
    return PP_ERR_ARG;
  }
  const float* src = (which ? m->vc : m->kc) + (size_t)layer * m->kv_layer_floats + (size_t)pos0 * row;
  PP_TRY(sync_model(m));
  PP_CUDA(cudaMemcpy(out, src, sizeof(float) * row * n_pos, cudaMemcpyDeviceToHost));
  return PP_OK;
}

int pp_get_stats(const pp_model* cm, pp_stats* out) {
  if (!cm || !out) return PP_ERR_ARG;
  pp_model* m = const_cast<pp_model*>(cm);
  PP_TRY(sync_model(m));
  PP_TRY(collect(m));
  *out = m->stats;
  const pp_config& c = m->cfg;
  out->kv_bytes = c.kv_grow ? (int64_t)m->kvs.mapped * m->kvs.n_regions
                            : (int64_t)2 * c.n_layers * c.max_seq * c.n_kv_heads * c.head_dim * (int64_t)sizeof(float);
  return PP_OK;
}

int pp_reset_stats(pp_model* m) {
  if (!m) return PP_ERR_ARG;
  PP_TRY(sync_model(m));
  PP_TRY(collect(m));
  m->stats = pp_stats{};
  m->lprof.assign(m->cfg.n_layers, pp_layer_profile{});
  return PP_OK;
}

int pp_set_chunk_overlap(pp_model* m, int32_t enable) {
  if (!m || (enable != 0 && enable != 1)) {
    set_err("bad pp_set_chunk_overlap arguments");
    return PP_ERR_ARG;
  }
  m->overlap = enable != 0;  // streams and scratch sets are made by the first call that needs them
  return PP_OK;
}

int pp_set_graphs(pp_model* m, int32_t enable) {
  if (!m || (enable != 0 && enable != 1)) {
    set_err("bad pp_set_graphs arguments");
    return PP_ERR_ARG;
  }
  if (!enable) {
    PP_TRY(sync_model(m));
    graphs_clear(m);
  }
  m->graphs = enable != 0;
  return PP_OK;
}

int pp_set_layer_profile(pp_model* m, int32_t enable) {
  if (!m || (enable != 0 && enable != 1)) {
    set_err("bad pp_set_layer_profile arguments");
    return PP_ERR_ARG;
  }
  PP_TRY(sync_model(m));
  PP_TRY(collect(m));
  if ((int)m->lprof.size() != m->cfg.n_layers) m->lprof.assign(m->cfg.n_layers, pp_layer_profile{});
  m->layer_prof = enable != 0;
  return PP_OK;
}

int pp_get_layer_profile(const pp_model* cm, pp_layer_profile* out, int32_t n_layers) {
  if (!cm || !out || n_layers != cm->cfg.n_layers) {
    set_err("bad pp_get_layer_profile arguments (n_layers must equal the model's)");
    return PP_ERR_ARG;
  }
  pp_model* m = const_cast<pp_model*>(cm);
  PP_TRY(sync_model(m));
  PP_TRY(collect(m));
  if ((int)m->lprof.size() != m->cfg.n_layers) m->lprof.assign(m->cfg.n_layers, pp_layer_profile{});
  for (int l = 0; l < n_layers; ++l) out[l] = m->lprof[l];
  return PP_OK;
}

int pp_model_gemm_engine(const pp_model* m) { return m ? m->engine : PP_ERR_ARG; }

int pp_set_trace(pp_model* m, float* d_x, int8_t* d_codes, float* d_scales, int32_t max_pos) {
  if (!m || (d_x && max_pos <= 0)) {
    set_err("bad pp_set_trace arguments");
    return PP_ERR_ARG;
  }
  PP_TRY(sync_model(m));
  m->trace = d_x;
  m->trace_codes = d_x ? d_codes : nullptr;
  m->trace_scales = d_x ? d_scales : nullptr;
  m->trace_pos = d_x ? max_pos : 0;
  return PP_OK;
}

int pp_set_profile_kernel(pp_model* m, int32_t kernel_class) {
  if (!m || kernel_class < PP_KERNEL_NONE || kernel_class >= PP_KERNEL_COUNT) {
    set_err("bad pp_set_profile_kernel arguments");
    return PP_ERR_ARG;
  }
  m->cfg.profile_kernel = kernel_class;
  return PP_OK;
}

// ---------------------------------------------------------------- single steps
static int ok_launch(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    set_err("%s: %s", what, cudaGetErrorString(e));
    return PP_ERR_CUDA;
  }
  return PP_OK;
}

int pp_op_quantize(const float* x, int32_t rows, int32_t k, int8_t* q8, uint16_t* q16, float* a_scale, void* stream) {
  if (!x || !q8 || !a_scale || rows <= 0 || k <= 0 || k % 4) { set_err("bad pp_op_quantize arguments"); return PP_ERR_ARG; }
  return ok_launch(launch_norm_quant(x, k, nullptr, rows, k, 0.f, nullptr, q8, reinterpret_cast<__half*>(q16), a_scale,
                                     static_cast<cudaStream_t>(stream)),
                   "quantize");
}

int pp_op_rmsnorm_quantize(const float* x, const float* g, int32_t rows, int32_t k, float eps, float* y_out, int8_t* q8,
                           uint16_t* q16, float* a_scale, void* stream) {
  if (!x || !g || !q8 || !a_scale || rows <= 0 || k <= 0 || k % 4 || eps < 0.f) {
    set_err("bad pp_op_rmsnorm_quantize arguments");
    return PP_ERR_ARG;
  }
  return ok_launch(launch_norm_quant(x, k, g, rows, k, eps, y_out, q8, reinterpret_cast<__half*>(q16), a_scale,
                                     static_cast<cudaStream_t>(stream)),
                   "rmsnorm_quantize");
}

static int check_gemm(int32_t engine, const int8_t* a8, const uint16_t* a16, const int8_t* w, int32_t m, int32_t n,
                      int32_t k) {
  if (!w || m <= 0 || n <= 0 || k <= 0 || k % 64 || n % 32) {
    set_err("bad GEMM shape m=%d n=%d k=%d (k%%64, n%%32)", m, n, k);
    return PP_ERR_ARG;
  }
  if (engine == PP_GEMM_MMA) {
    if (!a8) { set_err("the mma.sync engine needs the int8 activations"); return PP_ERR_ARG; }
    return PP_OK;
  }
  if (engine == PP_GEMM_TC) {
    if (!tc_available()) { set_err("the tcgen05 engine needs an sm_103 device"); return PP_ERR_UNSUPPORTED; }
    if (!a16 || n % 128 || (reinterpret_cast<uintptr_t>(a16) & 15) || (reinterpret_cast<uintptr_t>(w) & 15)) {
      set_err("the tcgen05 engine needs fp16 activations, n %% 128 == 0 and 16-byte aligned operands");
      return PP_ERR_ARG;
    }
    return PP_OK;
  }
  set_err("unknown gemm engine %d", engine);
  return PP_ERR_ARG;
}


// ---------------------------------------------------------------------------
// Device-side state of the single-step GEMM entry points that lives in this
// library's own device memory: the status word their bounded waits report to,
// and the fixed stream-K scratch of pp_op_gemm_noalloc (for callers that may
// not allocate device memory while they run: for example a host application
// that has already handed all device memory to its own pool allocator, or a
// latency-critical loop where cudaMalloc/cudaFree would block or synchronise
// the device). The CUDA runtime places these arrays on each device when the
// library's device code is loaded there; they stay until the process exits.
namespace {
constexpr size_t kStaticPartBytes = PP_NOALLOC_PART_BYTES;  // partial int32 tiles
constexpr int kStaticCounters = PP_NOALLOC_COUNTERS;        // per-tile arrival counters
static_assert(kStaticPartBytes % 256 == 0, "whole 256-byte lines");
static __device__ __align__(256) int32_t g_static_part[kStaticPartBytes / sizeof(int32_t)];
static __device__ __align__(256) int g_static_cnt[kStaticCounters];
static __device__ int g_op_status;  // DEV_OK or DEV_TIMEOUT, shared by every single-step GEMM call

struct StaticScratch {
  bool ready = false;
  int32_t* part = nullptr;
  int* cnt = nullptr;
  int* status = nullptr;
};
std::mutex g_static_mu;
StaticScratch g_static_dev[128];  // by device ordinal

// Device addresses of the arrays above on the current device. In host code the
// arrays' names stand for host-side shadows, not device addresses, so every
// pointer handed to a kernel comes from cudaGetSymbolAddress, looked up once per
// device (with that device current) on its first single-step GEMM call.
int static_scratch(StaticScratch* out) {
  int dev = 0;
  PP_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 128) {
    set_err("device ordinal %d out of range", dev);
    return PP_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticScratch& sc = g_static_dev[dev];
  if (!sc.ready) {
    void* part = nullptr;
    void* cnt = nullptr;
    void* st = nullptr;
    PP_CUDA(cudaGetSymbolAddress(&part, g_static_part));
    PP_CUDA(cudaGetSymbolAddress(&cnt, g_static_cnt));
    PP_CUDA(cudaGetSymbolAddress(&st, g_op_status));
    sc.part = static_cast<int32_t*>(part);
    sc.cnt = static_cast<int*>(cnt);
    sc.status = static_cast<int*>(st);
    sc.ready = true;
  }
  *out = sc;
  return PP_OK;
}

// Bounded waits of the single-step tcgen05 GEMMs (pp_debug_op_stall).
std::atomic<long long> g_op_wait_us{0};

TcWaits op_waits() {
  TcWaits w;
  const long long us = g_op_wait_us.load();
  if (us > 0) {
    int dev = 0, khz = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
    w.cycles = us * (khz > 0 ? khz : 2000000) / 1000;  // kHz -> cycles per microsecond
    w.hold_mma = 1;
  }
  return w;
}
}  // namespace

// One tcgen05 GEMM of a single-step entry point, with its tensor maps made for the
// call: k_gemm_tw for chunks of at most 128 rows, k_gemm_tc beyond (as in the model).
// Programmatic early start, but no weight load before griddepcontrol.wait: a caller's
// kernel may have written w just before the call.
static cudaError_t op_tc_launch(int epi, const uint16_t* a16, const int8_t* w, const float* ws, const float* as, int m,
                                int n, int k, float* out, int ldo, int32_t* acc, int* status, const TcWorkspace& wsp,
                                cudaStream_t st, const TcWaits& waits) {
  CUtensorMap ma, mw;
  const __half* a = reinterpret_cast<const __half*>(a16);
  cudaError_t e;
  if (m <= kTwMaxRows) {
    const int nt = tw_nt(m);
    if ((e = make_tmap_tw_tokens(&ma, a, m, k, nt)) != cudaSuccess) return e;
    if ((e = make_tmap_tw_weights(&mw, w, n, k)) != cudaSuccess) return e;
    return launch_gemm_tw(epi, ma, mw, nt, ws, as, m, n, k, out, ldo, acc, g_tc_seg.load(), status, wsp, st, waits,
                          TcRope{}, false, true, /*early_w=*/false);
  }
  const int bn = tc_bn(m, n, k);
  if ((e = make_tmap_a(&ma, a, m, k)) != cudaSuccess) return e;
  if ((e = make_tmap_w(&mw, w, n, k, bn)) != cudaSuccess) return e;
  return launch_gemm_tc(epi, ma, mw, bn, ws, as, m, n, k, out, ldo, acc, g_tc_seg.load(), status, wsp, st, waits,
                        TcRope{}, false, true, /*early_w=*/false);
}

// Process-wide stream-K workspace of pp_op_gemm / pp_op_gemm_acc, grown on
// demand (growing synchronises the device) and kept until exit.
static std::mutex g_op_ws_mu;
static TcWorkspace g_op_ws;

static cudaError_t op_workspace(int m, int n, int k, TcWorkspace* out) {
  size_t part = 0, cnt = 0;
  gemm_workspace_need(m, n, k, &part, &cnt);
  std::lock_guard<std::mutex> lk(g_op_ws_mu);
  if (part > g_op_ws.part_bytes || cnt > g_op_ws.counters) {
    if (g_op_ws.part) cudaFree(g_op_ws.part);
    if (g_op_ws.cnt) cudaFree(g_op_ws.cnt);
    g_op_ws = TcWorkspace{};
    const size_t pb = std::max(part, (size_t)256), cc = std::max(cnt, (size_t)64);
    cudaError_t e = cudaMalloc(&g_op_ws.part, pb);
    if (e != cudaSuccess) return e;
    e = cudaMalloc(&g_op_ws.cnt, cc * sizeof(int));
    if (e != cudaSuccess) return e;
    e = cudaMemset(g_op_ws.cnt, 0, cc * sizeof(int));
    if (e != cudaSuccess) return e;
    g_op_ws.part_bytes = pb;
    g_op_ws.counters = cc;
  }
  *out = g_op_ws;
  return cudaSuccess;
}

static int op_gemm_launch(int32_t engine, int epi, const int8_t* a8, const uint16_t* a16, const int8_t* w,
                          const float* ws, const float* as, int m, int n, int k, float* out, int ldo, int32_t* acc,
                          cudaStream_t st) {
  if (engine == PP_GEMM_MMA) return ok_launch(launch_gemm_mma(epi, a8, w, ws, as, m, n, k, out, ldo, acc, st), "gemm");
  StaticScratch sc;
  PP_TRY(static_scratch(&sc));
  TcWorkspace wsp;
  PP_CUDA(op_workspace(m, n, k, &wsp));
  return ok_launch(op_tc_launch(epi, a16, w, ws, as, m, n, k, out, ldo, acc, sc.status, wsp, st, op_waits()), "gemm");
}

int pp_op_gemm_acc(int32_t engine, const int8_t* a8, const uint16_t* a16, const int8_t* w, int32_t m, int32_t n,
                   int32_t k, int32_t* acc, void* stream) {
  PP_TRY(check_gemm(engine, a8, a16, w, m, n, k));
  if (!acc) { set_err("null acc"); return PP_ERR_ARG; }
  return op_gemm_launch(engine, EPI_ACC, a8, a16, w, nullptr, nullptr, m, n, k, nullptr, 0, acc,
                        static_cast<cudaStream_t>(stream));
}

int pp_op_gemm(int32_t engine, int32_t epilogue, const int8_t* a8, const uint16_t* a16, const int8_t* w,
               const float* w_scale, const float* a_scale, int32_t m, int32_t n, int32_t k, float* out, int32_t ldo,
               void* stream) {
  PP_TRY(check_gemm(engine, a8, a16, w, m, n, k));
  if (engine == PP_GEMM_TC && (reinterpret_cast<uintptr_t>(w_scale) & 15)) {
    set_err("the tcgen05 engine needs 16-byte aligned row scales");
    return PP_ERR_ARG;
  }
  const int out_cols = epilogue == PP_EPI_SWIGLU ? n / 2 : n;
  if (!w_scale || !a_scale || !out || ldo < out_cols || (epilogue < PP_EPI_STORE || epilogue > PP_EPI_SWIGLU) ||
      ldo % 4 || (reinterpret_cast<uintptr_t>(out) & 15)) {
    set_err("bad pp_op_gemm arguments (ldo %% 4, 16-byte aligned out)");
    return PP_ERR_ARG;
  }
  return op_gemm_launch(engine, epilogue, a8, a16, w, w_scale, a_scale, m, n, k, out, ldo, nullptr,
                        static_cast<cudaStream_t>(stream));
}

int pp_op_status(void* stream) {
  StaticScratch sc;
  PP_TRY(static_scratch(&sc));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  PP_CUDA(cudaMemcpyAsync(&v, sc.status, sizeof(int), cudaMemcpyDeviceToHost, st));
  PP_CUDA(cudaStreamSynchronize(st));
  if (v == DEV_OK) return PP_OK;
  PP_CUDA(cudaMemsetAsync(sc.status, 0, sizeof(int), st));
  {
    // a call that gave up can leave stream-K arrival counters behind
    std::lock_guard<std::mutex> lk(g_op_ws_mu);
    if (g_op_ws.cnt) PP_CUDA(cudaMemsetAsync(g_op_ws.cnt, 0, g_op_ws.counters * sizeof(int), st));
  }
  PP_CUDA(cudaStreamSynchronize(st));
  set_err("a bounded device wait of a single-step GEMM gave up");
  return PP_ERR_DEVICE_TIMEOUT;
}


// ---------------------------------------------------------------- host-buffer checks
int pp_debug_quantize(const float* x, int32_t rows, int32_t k, int8_t* q, float* a_scale) {
  if (!x || !q || !a_scale || rows <= 0 || k <= 0 || k % 4) {
    set_err("bad pp_debug_quantize arguments");
    return PP_ERR_ARG;
  }
  const size_t n = (size_t)rows * k;
  DeviceScratch d;
  float *dx = nullptr, *ds = nullptr;
  int8_t* dq = nullptr;
  PP_TRY(d.upload(&dx, x, n));
  PP_TRY(d.alloc(&dq, n));
  PP_TRY(d.alloc(&ds, (size_t)rows));
  PP_TRY(pp_op_quantize(dx, rows, k, dq, nullptr, ds, nullptr));
  PP_CUDA(cudaMemcpy(q, dq, n, cudaMemcpyDeviceToHost));
  PP_CUDA(cudaMemcpy(a_scale, ds, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost));
  return PP_OK;
}

int pp_debug_gemm_i8(const int8_t* a, const int8_t* w, int32_t m, int32_t n, int32_t k, int32_t* acc) {
  if (!acc) {
    set_err("null acc");
    return PP_ERR_ARG;
  }
  return debug_gemm(a, w, nullptr, nullptr, nullptr, m, n, k, acc, nullptr);
}

int pp_debug_gemm_epilogue(const int8_t* a, const int8_t* w, const float* w_scale, const float* a_scale,
                           const float* resid, int32_t m, int32_t n, int32_t k, float* out) {
  if (!out) {
    set_err("null out");
    return PP_ERR_ARG;
  }
  return debug_gemm(a, w, w_scale, a_scale, resid, m, n, k, nullptr, out);
}

int pp_debug_op_stall(int32_t wait_us) {
  if (wait_us < 0) {
    set_err("bad pp_debug_op_stall arguments");
    return PP_ERR_ARG;
  }
  g_op_wait_us.store(wait_us);
  return PP_OK;
}

int pp_op_gemm_noalloc_need(int32_t m, int32_t n, int32_t k, int64_t* part_bytes, int64_t* counters) {
  if (!part_bytes || !counters || m <= 0 || n <= 0 || k <= 0 || k % 64 || n % 128) {
    set_err("bad pp_op_gemm_noalloc_need arguments (k %% 64, n %% 128)");
    return PP_ERR_ARG;
  }
  if (!tc_available()) {
    set_err("the tcgen05 engine needs an sm_103 device");
    return PP_ERR_UNSUPPORTED;
  }
  size_t pb = 0, cc = 0;
  gemm_workspace_need(m, n, k, &pb, &cc);
  *part_bytes = (int64_t)pb;
  *counters = (int64_t)cc;
  return PP_OK;
}

int pp_op_gemm_noalloc(int32_t epilogue, const uint16_t* a16, const int8_t* w, const float* w_scale,
                       const float* a_scale, int32_t m, int32_t n, int32_t k, float* out, int32_t ldo, void* stream) {
  PP_TRY(check_gemm(PP_GEMM_TC, nullptr, a16, w, m, n, k));
  const int out_cols = epilogue == PP_EPI_SWIGLU ? n / 2 : n;
  if (!w_scale || !a_scale || !out || ldo < out_cols || (epilogue < PP_EPI_STORE || epilogue > PP_EPI_SWIGLU) ||
      ldo % 4 || (reinterpret_cast<uintptr_t>(out) & 15) || (reinterpret_cast<uintptr_t>(w_scale) & 15)) {
    set_err("bad pp_op_gemm_noalloc arguments");
    return PP_ERR_ARG;
  }
  size_t need_part = 0, need_cnt = 0;
  gemm_workspace_need(m, n, k, &need_part, &need_cnt);
  if (need_part > kStaticPartBytes || need_cnt > (size_t)kStaticCounters) {
    set_err("GEMM m=%d n=%d k=%d needs %zu bytes of scratch and %zu counters; the fixed scratch holds %zu bytes and %d",
            m, n, k, need_part, need_cnt, kStaticPartBytes, kStaticCounters);
    return PP_ERR_ARG;
  }
  StaticScratch sc;
  PP_TRY(static_scratch(&sc));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: counters must start at zero
  if (need_cnt) PP_CUDA(cudaMemsetAsync(sc.cnt, 0, need_cnt * sizeof(int), st));
  TcWorkspace wsp;
  wsp.part = sc.part;
  wsp.part_bytes = kStaticPartBytes;
  wsp.cnt = sc.cnt;
  wsp.counters = kStaticCounters;
  return ok_launch(op_tc_launch(epilogue, a16, w, w_scale, a_scale, m, n, k, out, ldo, nullptr, sc.status, wsp, st,
                                op_waits()),
                   "gemm_noalloc");
}

int pp_debug_noalloc_poison(int32_t value) {
  StaticScratch sc;
  PP_TRY(static_scratch(&sc));
  std::vector<int> v(kStaticCounters, value);
  PP_CUDA(cudaMemcpy(sc.cnt, v.data(), v.size() * sizeof(int), cudaMemcpyHostToDevice));
  return PP_OK;
}

int pp_set_exact_segment(int32_t seg_k) {
  if (seg_k < 64 || seg_k > kTcSegK || seg_k % 64) {
    set_err("exact segment must be a multiple of 64 in [64, %d]", kTcSegK);
    return PP_ERR_ARG;
  }
  g_tc_seg.store(seg_k);
  return PP_OK;
}

int pp_debug_gemm_stall(int32_t wait_us, const uint16_t* a16, const int8_t* w, int32_t m, int32_t n, int32_t k,
                        int32_t* acc) {
  if (wait_us <= 0 || !acc) {
    set_err("bad pp_debug_gemm_stall arguments");
    return PP_ERR_ARG;
  }
  PP_TRY(check_gemm(PP_GEMM_TC, nullptr, a16, w, m, n, k));
  int dev = 0, khz = 0;
  PP_CUDA(cudaGetDevice(&dev));
  PP_CUDA(cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev));
  int* status = nullptr;
  PP_CUDA(cudaMalloc(&status, sizeof(int)));
  cudaError_t e = cudaMemset(status, 0, sizeof(int));
  TcWaits waits;
  waits.cycles = (long long)wait_us * (khz > 0 ? khz : 2000000) / 1000;  // kHz -> cycles per microsecond
  waits.hold_mma = 1;
  if (e == cudaSuccess)  // no stream-K workspace: whole tiles, no counters left behind
    e = op_tc_launch(EPI_ACC, a16, w, nullptr, nullptr, m, n, k, nullptr, n, acc, status, TcWorkspace{}, nullptr, waits);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(status);
  if (e != cudaSuccess) {
    set_err("pp_debug_gemm_stall: %s", cudaGetErrorString(e));
    return PP_ERR_CUDA;
  }
  if (st == DEV_TIMEOUT) {
    set_err("a bounded device wait gave up (held-back MMA issuer)");
    return PP_ERR_DEVICE_TIMEOUT;
  }
  return PP_OK;
}

int pp_debug_loader_fault(pp_model* m, int32_t fault) {
  if (!m || (fault != 0 && fault != 1)) {
    set_err("bad pp_debug_loader_fault arguments");
    return PP_ERR_ARG;
  }
  PP_TRY(sync_model(m));
  m->loader_fault = fault;
  return PP_OK;
}

int pp_debug_alloc_cap(int64_t bytes) {
  if (bytes < 0) {
    set_err("bad pp_debug_alloc_cap arguments");
    return PP_ERR_ARG;
  }
  g_alloc_cap.store(bytes);
  return PP_OK;
}

int pp_op_rope_table(int32_t max_pos, int32_t head_dim, float theta, float* rope_table, void* stream) {
  if (max_pos <= 0 || head_dim <= 0 || head_dim % 2 || theta <= 0.f || !rope_table) {
    set_err("bad pp_op_rope_table arguments");
    return PP_ERR_ARG;
  }
  return ok_launch(launch_rope_table(max_pos, head_dim, theta, rope_table, static_cast<cudaStream_t>(stream)),
                   "rope_table");
}

int pp_op_rope_kv(const float* qkv, int32_t rows, int32_t start_pos, int32_t n_heads, int32_t n_kv_heads,
                  int32_t head_dim, const float* rope_table, float* q_out, float* k_cache, float* v_cache,
                  void* stream) {
  if (!qkv || !rope_table || !q_out || !k_cache || !v_cache || rows <= 0 || start_pos < 0 || n_heads <= 0 ||
      n_kv_heads <= 0 || head_dim <= 0 || head_dim % 2) {
    set_err("bad pp_op_rope_kv arguments");
    return PP_ERR_ARG;
  }
  return ok_launch(launch_rope_kv(qkv, rows, start_pos, n_heads, n_kv_heads, head_dim, rope_table, q_out, k_cache,
                                  v_cache, static_cast<cudaStream_t>(stream)),
                   "rope_kv");
}

// Per-key-range partial state of the single-step attention entry point,
// grown on demand and kept until exit; calls are serialised by the mutex
// only on the host, so concurrent calls on different streams would share it.
static std::mutex g_attn_ws_mu;
static float* g_attn_ws = nullptr;
static size_t g_attn_ws_bytes = 0;

int pp_op_attention(const float* q, const float* k_cache, const float* v_cache, int32_t rows, int32_t start_pos,
                    int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float* o, void* stream) {
  if (!q || !k_cache || !v_cache || !o || rows <= 0 || start_pos < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
      n_heads % n_kv_heads || 64 % (n_heads / n_kv_heads) || (head_dim != 64 && head_dim != 128)) {
    set_err("bad pp_op_attention arguments");
    return PP_ERR_ARG;
  }
  const size_t need = attention_workspace_bytes(rows, start_pos, n_heads, n_kv_heads, head_dim);
  std::lock_guard<std::mutex> lk(g_attn_ws_mu);
  if (need > g_attn_ws_bytes) {
    // grow the process-wide range workspace (cudaFree waits for the device)
    if (g_attn_ws) cudaFree(g_attn_ws);
    g_attn_ws = nullptr;
    g_attn_ws_bytes = 0;
    cudaError_t e = cudaMalloc(&g_attn_ws, need);
    if (e != cudaSuccess) return ok_launch(e, "attention workspace");
    g_attn_ws_bytes = need;
  }
  return ok_launch(launch_attention(q, k_cache, v_cache, rows, start_pos, n_heads, n_kv_heads, head_dim, o,
                                    g_attn_ws, g_attn_ws_bytes, static_cast<cudaStream_t>(stream)),
                   "attention");
}

int pp_op_lm_head(const int8_t* q8, const float* a_scale, const int8_t* w_out, const float* w_scale, int32_t vocab,
                  int32_t dim, float* logits, void* stream) {
  if (!q8 || !a_scale || !w_out || !w_scale || !logits || vocab <= 0 || dim <= 0 || dim % 16 ||
      (reinterpret_cast<uintptr_t>(q8) & 15) || (reinterpret_cast<uintptr_t>(w_out) & 15)) {
    set_err("bad pp_op_lm_head arguments (dim%%16, 16-byte aligned int8 buffers)");
    return PP_ERR_ARG;
  }
  return ok_launch(launch_lm_head(q8, a_scale, w_out, w_scale, vocab, dim, logits, static_cast<cudaStream_t>(stream)),
                   "lm_head");
}

}  // extern "C"
