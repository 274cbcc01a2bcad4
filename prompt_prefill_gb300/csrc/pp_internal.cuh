// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include <cstdint>

#include "pp.h"

namespace pp {

// Host-side facts kept per device (a kernel's shared-memory attribute set, occupancy
// counts): one slot per device ordinal below kMaxDevices, recomputed on every call above.
constexpr int kMaxDevices = 64;

// Runs `set` (returning cudaError_t) on the current device until it has succeeded once there.
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < kMaxDevices ? (uint64_t)1 << dev : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// The positive int `get()` computes for the current device, computed once per device.
template <typename F>
int per_device(std::atomic<int> (&cache)[kMaxDevices], F&& get) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return get();
  int v = cache[dev].load(std::memory_order_acquire);
  if (v <= 0) {
    v = get();
    cache[dev].store(v, std::memory_order_release);
  }
  return v;
}

// Epilogue selector of the GEMM kernels (PP_EPI_* plus the raw int32 form).
// EPI_ROPE (tcgen05 engine only): RoPE + K/V write of a QKV projection whose q and k
// head rows are in pair order (see TcRope).
enum Epi : int { EPI_STORE = PP_EPI_STORE, EPI_RESID = PP_EPI_RESID, EPI_SWIGLU = PP_EPI_SWIGLU, EPI_ACC = 3, EPI_ROPE = 4 };

// Device status word values (written by kernels, read by pp_device_status).
enum : int { DEV_OK = 0, DEV_BAD_TOKEN = 1, DEV_TIMEOUT = 2 };

// ---- elementwise / row kernels (k_rows.cu)
// pdl (every launcher below that takes it): allow the launch to start early behind the
// stream's previous kernel (programmatic dependent launch); false gives a plain
// stream-ordered launch, for the first kernel after a wait on another stream's event.
cudaError_t launch_embed(const int32_t* tok, int n, const float* emb, int vocab, int dim, float* x, int* status,
                         cudaStream_t s, bool pdl = true);
cudaError_t launch_norm_quant(const float* x, int ldx, const float* g, int rows, int k, float eps, float* y,
                              int8_t* q8, __half* q16, float* a_scale, cudaStream_t s, bool pdl = true);
cudaError_t launch_rope_table(int max_pos, int hd, float theta, float* table, cudaStream_t s);
// a [n] int8 -> out [n] fp16, exact.
cudaError_t launch_widen_i8(const int8_t* a, long long n, __half* out, cudaStream_t s);
// paired: the q and k head columns of qkv are in pair order (dims j and j + hd/2 at
// columns 2j and 2j + 1 of the head), as the model's packed QKV weights produce them.
cudaError_t launch_rope_kv(const float* qkv, int rows, int start_pos, int H, int Hkv, int hd, const float* table,
                           float* q_out, float* k_cache, float* v_cache, cudaStream_t s, bool paired = false,
                           bool pdl = true);
cudaError_t launch_lm_head(const int8_t* q8, const float* a_scale, const int8_t* w, const float* ws, int vocab,
                           int dim, float* logits, cudaStream_t s, bool pdl = true);

// ---- GEMMs
// mma.sync engine (k_gemm_mma.cu): a8 [m][k] int8, w [n][k] int8.
cudaError_t launch_gemm_mma(int epi, const int8_t* a8, const int8_t* w, const float* ws, const float* as, int m,
                            int n, int k, float* out, int ldo, int32_t* acc, cudaStream_t s);

// tcgen05 engine (k_gemm_tc.cu): a16 [m][k] fp16 codes via a tensor map, w [n][k] int8 via a tensor map.
// n % 128 == 0, k % 64 == 0; exact f32 segments of seg_k (<= 1024) along k. The weight map's box
// is made for one tile width bn (256, 192 or 128): the one tc_bn(m, n, k) picks for the launch.
bool tc_available();
constexpr int kTcBn[3] = {256, 192, 128};
// wide: the widest width that divides n and no stream-K (for launches whose idle
// CTA pairs other streams fill).
int tc_bn(int m, int n, int k, bool wide = false);
inline int tc_bn_index(int m, int n, int k, bool wide = false) {
  const int bn = tc_bn(m, n, k, wide);
  return bn == 256 ? 0 : (bn == 192 ? 1 : 2);
}
cudaError_t make_tmap_a(CUtensorMap* map, const __half* a16, int rows, int k);
cudaError_t make_tmap_w(CUtensorMap* map, const int8_t* w, int n, int k, int bn);
// Stream-K workspace: int32 partial tiles and per-tile counters (zero between launches).
struct TcWorkspace {
  int32_t* part = nullptr;
  size_t part_bytes = 0;
  int* cnt = nullptr;
  size_t counters = 0;
};
// Workspace a GEMM of this shape uses (0 when it runs whole tiles).
void tc_workspace_need(int m, int n, int k, size_t* part_bytes, size_t* counters);
// Bound of every mbarrier wait in the tcgen05 GEMM (on expiry: DEV_TIMEOUT in the status word, the kernel
// lets its copies and MMAs land, frees its TMEM and exits), and a test hook that holds back the MMA issuer.
struct TcWaits {
  long long cycles = 4000000000LL;  // ~2 s at 2 GHz
  int hold_mma = 0;
};
// EPI_ROPE destinations: the GEMM's n = (H + 2 Hkv) hd columns are q heads, k heads, v heads,
// with the rows of every q and k head in pair order; row r of the GEMM is position pos0 + r.
struct TcRope {
  const float* table = nullptr;  // [max_pos][hd/2] (cos, sin)
  int pos0 = 0, H = 0, Hkv = 0, hd = 0;
  float* q_out = nullptr;    // [m][H][hd]
  float* k_cache = nullptr;  // [pos][Hkv][hd]
  float* v_cache = nullptr;  // [pos][Hkv][hd]
};
// early_w: the producer may load the first pipeline stages' weights before its
// griddepcontrol.wait, i.e. while the stream's previous kernel still runs. Only
// for weights that no kernel of the stream writes (the model's own weight blocks;
// a streamed layer's ring slot is waited for with a plain launch first); the
// single-step entry points leave it off, so a caller's kernel that writes w just
// before the call is always seen.
cudaError_t launch_gemm_tc(int epi, const CUtensorMap& ma, const CUtensorMap& mw, int bn, const float* ws,
                           const float* as, int m, int n, int k, float* out, int ldo, int32_t* acc, int seg_k,
                           int* status, const TcWorkspace& wsp, cudaStream_t s, const TcWaits& waits = TcWaits{},
                           const TcRope& rope = TcRope{}, bool wide = false, bool pdl = true, bool early_w = false);
constexpr int kTcSegK = 1024;  // 1024 * 127^2 < 2^24: every f32 partial sum of a segment is an exact integer

// tcgen05 engine for chunks of at most 128 rows (k_gemm_tw.cu): the weights are the MMA's M side
// (256 weight rows per CTA pair, converted into tensor memory) and the chunk's tokens its N side
// (NT = tw_nt(m) = 32, 64 or 128). Same operands, segments, workspace, waits and epilogues as
// launch_gemm_tc; the token map's box is made for one NT, the weight map for every launch.
constexpr int kTwNt[3] = {128, 64, 32};
constexpr int kTwMaxRows = 128;
int tw_nt(int m);
inline int tw_nt_index(int m) {
  const int nt = tw_nt(m);
  return nt == 128 ? 0 : (nt == 64 ? 1 : 2);
}
cudaError_t make_tmap_tw_tokens(CUtensorMap* map, const __half* a16, int rows, int k, int nt);
cudaError_t make_tmap_tw_weights(CUtensorMap* map, const int8_t* w, int n, int k);
void tw_workspace_need(int m, int n, int k, size_t* part_bytes, size_t* counters);
cudaError_t launch_gemm_tw(int epi, const CUtensorMap& mt, const CUtensorMap& mw, int nt, const float* ws,
                           const float* as, int m, int n, int k, float* out, int ldo, int32_t* acc, int seg_k,
                           int* status, const TcWorkspace& wsp, cudaStream_t s, const TcWaits& waits = TcWaits{},
                           const TcRope& rope = TcRope{}, bool wide = false, bool pdl = true, bool early_w = false);

// ---- attention (k_attention.cu)
// Keys per range of the attention work split, at fixed absolute positions.
constexpr int kAttnRange = 512;
// Bytes of per-range partial state a launch of this size needs (0: one range).
size_t attention_workspace_bytes(int rows, int start_pos, int H, int Hkv, int hd);
// pdl: allow the launch to start early behind the stream's previous kernel
// (off when another stream's event must hold it back).
cudaError_t launch_attention(const float* q, const float* kc, const float* vc, int rows, int start_pos, int H,
                             int Hkv, int hd, float* o, float* part, size_t part_bytes, cudaStream_t s,
                             bool pdl = true);

// ---- grow-on-demand K/V memory (kv_space.cu): n_regions regions of region_bytes
// in one reserved virtual range; the first `mapped` bytes of every region are
// backed by device memory. The caller synchronises before kv_space_release.
struct KvSpace {
  unsigned long long base = 0;  // CUdeviceptr of the reserved range
  size_t gran = 0, region_bytes = 0, mapped = 0;
  int n_regions = 0, device = 0;
  struct Map {
    unsigned long long ptr;
    size_t size;
    unsigned long long handle;
  };
  std::vector<Map> maps;
};
cudaError_t kv_space_reserve(KvSpace* s, int device, int n_regions, size_t region_min_bytes);
cudaError_t kv_space_grow(KvSpace* s, size_t region_bytes_needed);
void kv_space_release(KvSpace* s);
void kv_space_free(KvSpace* s);

// Rows of the interleaved gate/up matrix: blocks of 16 gate rows then 16 up rows.
constexpr int kSwiGluBlock = 16;

// Launch kern<<<grid, block, smem, s>>>(args...) with programmatic dependent
// launch allowed (the kernel calls ppdev::pdl_wait before using its inputs),
// or as a plain stream-ordered launch when pdl is false.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_if(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  return launch_pdl_if(true, kern, grid, block, smem, s, args...);
}

}  // namespace pp

// ---------------------------------------------------------------- PTX helpers
namespace ppdev {

// Programmatic dependent launch: a kernel launched with launch_pdl may start
// while the previous kernel of its stream is still running. pdl_trigger lets
// this kernel's own dependents be scheduled; pdl_wait blocks until every
// earlier kernel of the stream has finished and its writes are visible, and
// must come before the first read of their results (and the first write of
// anything they read). Both are no-ops for a kernel launched without it.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D = A(16x32 s8, row) * B(32x8 s8, col) + D, int32 accumulate (exact).
__device__ __forceinline__ void mma_s8_16832(int32_t (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// The dequantising epilogue in its fixed order: (float(acc) * w_scale) * a_scale,
// each product rounded to nearest (no contraction).
__device__ __forceinline__ float dequant(int32_t acc, float ws, float as) {
  return __fmul_rn(__fmul_rn(__int2float_rn(acc), ws), as);
}

// RoPE rotation of the pair (a, b) = (x_j, x_{j + hd/2}) by (c, s) = (cos, sin):
// (a c - b s, a s + b c), each a fused multiply-add of one rounded product, in
// this fixed form wherever the model rotates (the GEMM epilogue and the RoPE kernel).
__device__ __forceinline__ float2 rope_rot(float a, float b, float2 cs) {
  return make_float2(__fmaf_rn(a, cs.x, -__fmul_rn(b, cs.y)), __fmaf_rn(a, cs.y, __fmul_rn(b, cs.x)));
}

// SwiGLU gate: silu(g) * u = (g / (1 + exp(-g))) * u in f32, each step rounded to
// nearest: CUDA's full-accuracy expf (at most 2 ulp), an IEEE add, an IEEE division
// and an IEEE multiply, so the result is within a few ulp of the exact value. For
// g < -88.7 exp(-g) overflows to inf and the gate gives -0 where the exact value is a
// subnormal of magnitude below 2^-126 * |g|.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

}  // namespace ppdev
