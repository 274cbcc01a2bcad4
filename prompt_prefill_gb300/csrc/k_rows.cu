// Row-wise kernels of the prefill path: embedding gather, RMSNorm + per-token
// int8 quantiser, RoPE table and RoPE + K/V write, and the last-position
// output projection. All are HBM/L2-bound; each keeps every per-row reduction
// in one fixed order so that a row's result never depends on which other rows
// share its launch (the chunk size).
#include <cfloat>

#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int kRowThreads = 256;

// Embedding gather ("Single-pass prefill": prefill runs the prompt through the
// model): x[i] = emb[tok[i]]. Ids outside [0, vocab) give a zero row and set
// the device status word.
__global__ void __launch_bounds__(kRowThreads) k_embed(const int32_t* __restrict__ tok, const float* __restrict__ emb,
                                                     int vocab, int dim, float* __restrict__ x, int* status) {
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  const int i = blockIdx.x;
  const int t = tok[i];
  const bool ok = t >= 0 && t < vocab;
  if (!ok && threadIdx.x == 0 && status) atomicCAS(status, DEV_OK, DEV_BAD_TOKEN);
  const float4* src = reinterpret_cast<const float4*>(emb + (size_t)(ok ? t : 0) * dim);
  float4* dst = reinterpret_cast<float4*>(x + (size_t)i * dim);
  for (int c = threadIdx.x; c < dim / 4; c += kRowThreads) dst[c] = ok ? __ldg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Fixed-order block reductions: per-thread partials, xor butterfly within a
// warp, then every thread folds the warp results in index order (one barrier;
// each reduction of a kernel uses its own `red` array, so none is reused).
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) s += red[i];
  return s;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) m = fmaxf(m, red[i]);
  return m;
}

// Maximum that returns NaN when either operand is NaN (fmaxf ignores a NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ float block_max_nan(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) m = max_nan(m, red[i]);
  return m;
}

// Codes by IEEE addition. For a finite row with amax > 0 and inv = 127/amax
// finite, every v = y * inv has |v| <= 127 (1 + 2^-24)^2 < 127.5, so the
// clamp of the quantiser never acts. kCodeMagic = 1.5 * 2^23 + 0x6600 is an
// even integer in [2^23, 2^24), where the f32 grid is the integers: the
// round-to-nearest-even sum kCodeMagic + v is exactly kCodeMagic + q with
// q = rint_even(v), so its low 16 bits are 0x6600 + q, the fp16 bits of
// 1536 + q (fp16 spacing is 1 on [1024, 2048)), and its low byte is q in two's
// complement. Two sums give a half2 of 1536 + q by one byte permute; the fp16
// subtraction of 1536 is exact (Sterbenz), leaving q. No conversion instruction
// is needed.
constexpr float kCodeMagic = 12609024.0f;  // 0x4B406600

struct Codes4 {
  uint32_t q8;  // four int8 codes
  uint2 q16;    // four fp16 codes
};

__device__ __forceinline__ Codes4 codes_fast(const float y[4], float inv) {
  uint32_t u[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) u[e] = __float_as_uint(__fadd_rn(__fmul_rn(y[e], inv), kCodeMagic));
  const uint32_t h01 = __byte_perm(u[0], u[1], 0x5410), h23 = __byte_perm(u[2], u[3], 0x5410);
  const __half2 off = __float2half2_rn(1536.0f);
  __half2 a = *reinterpret_cast<const __half2*>(&h01), b = *reinterpret_cast<const __half2*>(&h23);
  a = __hsub2(a, off);
  b = __hsub2(b, off);
  Codes4 c;
  c.q8 = __byte_perm(h01, h23, 0x6420);
  c.q16 = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  return c;
}

// The quantiser's definition written out, for rows the fast form does not
// cover (a non-finite element, or amax so small that 127/amax overflows).
__device__ __forceinline__ Codes4 codes_exact(const float y[4], float inv, bool zero) {
  int qi[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int q = zero ? 0 : __float2int_rn(__fmul_rn(y[e], inv));
    qi[e] = q > 127 ? 127 : (q < -127 ? -127 : q);
  }
  Codes4 c;
  c.q8 = (uint32_t)(uint8_t)qi[0] | (uint32_t)(uint8_t)qi[1] << 8 | (uint32_t)(uint8_t)qi[2] << 16 |
         (uint32_t)(uint8_t)qi[3] << 24;
  const __half2 a = __halves2half2(__int2half_rn(qi[0]), __int2half_rn(qi[1]));
  const __half2 b = __halves2half2(__int2half_rn(qi[2]), __int2half_rn(qi[3]));
  c.q16 = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  return c;
}

// RMSNorm (optional) then the per-token absmax quantiser ("Batched Prefill",
// "The Solution": quantise each token once per chunk; every output row reuses
// the codes). One CTA per row:
//   r = 1 / sqrt(sum(x^2)/k + eps), y = (x * r) * g            (NORM only)
//   amax = max|y|, inv = 127/amax, q = clamp(rint_even(y*inv), +-127), a_scale = amax/127
// All f32 with IEEE division and square root; amax == 0 gives q = 0, a_scale = 0.
// amax is reduced with a NaN-propagating maximum: a finite row whose inv is
// finite takes the conversion-free codes (codes_fast); any other row (NaN or
// infinity in it, or a tiny amax) recomputes amax ignoring NaN and takes the
// written-out definition, a branch uniform over the CTA. Both give the same
// codes wherever both apply.
// NV > 0: the thread's NV float4 of the row are loaded once and kept in
// registers for all passes (k <= 4 * NV * kRowThreads), and for NV <= 4 the
// thread's norm weights are loaded with them; NV == 0 streams the row from
// memory in each pass (any k). Every pass visits the thread's elements in the
// same order, so all forms give the same bits. q8 or q16 may be null (that copy
// of the codes is not written).
template <bool NORM, int NV>
__global__ void __launch_bounds__(kRowThreads)
    k_norm_quant(const float* __restrict__ x, int ldx, const float* __restrict__ g, int k, float eps,
                 float* __restrict__ y_out, int8_t* __restrict__ q8, __half* __restrict__ q16,
                 float* __restrict__ a_scale) {
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  __shared__ float red_sum[kRowThreads / 32], red_max[kRowThreads / 32], red_max2[kRowThreads / 32];
  const int row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * ldx);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const int k4 = k >> 2;
  constexpr int NR = NV > 0 ? NV : 1;
  constexpr bool GPRE = NORM && NV > 0 && NV <= 4;  // norm weights held in registers too
  constexpr int NG = GPRE ? NR : 1;
  float4 xv[NR], gv[NG];
  if (NV > 0) {
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int c = threadIdx.x + j * kRowThreads;
      if (c < k4) xv[j] = xr[c];
    }
  }
  if (GPRE) {
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int c = threadIdx.x + j * kRowThreads;
      if (c < k4) gv[j] = __ldg(g4 + c);
    }
  }
  // f(x[4c .. 4c+3], g[4c .. 4c+3], c) for this thread's c in increasing order
  auto for_each = [&](auto&& f) {
    if (NV > 0) {
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        const int c = threadIdx.x + j * kRowThreads;
        if (c < k4) f(xv[j], GPRE ? gv[GPRE ? j : 0] : (NORM ? __ldg(g4 + c) : make_float4(1.f, 1.f, 1.f, 1.f)), c);
      }
    } else {
      for (int c = threadIdx.x; c < k4; c += kRowThreads)
        f(xr[c], NORM ? __ldg(g4 + c) : make_float4(1.f, 1.f, 1.f, 1.f), c);
    }
  };
  float r = 1.f;
  if (NORM) {
    float ss = 0.f;
    for_each([&](const float4& v, const float4&, int) {
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    });
    ss = block_sum(ss, red_sum);
    r = 1.0f / sqrtf(ss / (float)k + eps);
  }
  auto yval = [&](float xv_, float gv_) { return NORM ? __fmul_rn(__fmul_rn(xv_, r), gv_) : xv_; };
  float amax = 0.f;
  for_each([&](const float4& v, const float4& gg, int) {
    amax = max_nan(amax, fabsf(yval(v.x, gg.x)));
    amax = max_nan(amax, fabsf(yval(v.y, gg.y)));
    amax = max_nan(amax, fabsf(yval(v.z, gg.z)));
    amax = max_nan(amax, fabsf(yval(v.w, gg.w)));
  });
  amax = block_max_nan(amax, red_max);
  float inv = amax == 0.f ? 0.f : 127.0f / amax;
  const bool fast = amax <= FLT_MAX && inv <= FLT_MAX;  // false for NaN and infinity
  if (!fast) {  // uniform over the CTA: amax as the definition takes it, NaN ignored
    amax = 0.f;
    for_each([&](const float4& v, const float4& gg, int) {
      amax = fmaxf(amax, fabsf(yval(v.x, gg.x)));
      amax = fmaxf(amax, fabsf(yval(v.y, gg.y)));
      amax = fmaxf(amax, fabsf(yval(v.z, gg.z)));
      amax = fmaxf(amax, fabsf(yval(v.w, gg.w)));
    });
    amax = block_max(amax, red_max2);
    inv = amax == 0.f ? 0.f : 127.0f / amax;
  }
  const bool zero = amax == 0.f;
  for_each([&](const float4& v, const float4& gg, int c) {
    const float y[4] = {yval(v.x, gg.x), yval(v.y, gg.y), yval(v.z, gg.z), yval(v.w, gg.w)};
    const Codes4 q = fast ? codes_fast(y, inv) : codes_exact(y, inv, zero);
    const size_t base = (size_t)row * k + 4 * (size_t)c;
    if (q8) *reinterpret_cast<uint32_t*>(q8 + base) = q.q8;
    if (q16) *reinterpret_cast<uint2*>(q16 + base) = q.q16;
    if (y_out) reinterpret_cast<float4*>(y_out + base)[0] = make_float4(y[0], y[1], y[2], y[3]);
  });
  if (threadIdx.x == 0) a_scale[row] = zero ? 0.f : amax / 127.0f;
}

// RoPE table: table[pos][j] = (cos, sin)(pos * theta^(-2j/hd)), angles in double.
__global__ void k_rope_table(int max_pos, int hd, double theta, float2* __restrict__ table) {
  const int half = hd / 2;
  const long long n = (long long)max_pos * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(e / half), j = (int)(e % half);
    const double freq = pow(theta, -2.0 * (double)j / (double)hd);
    double s, c;
    sincos((double)pos * freq, &s, &c);
    table[e] = make_float2((float)c, (float)s);
  }
}

// RoPE + K/V write ("Single-pass prefill": K/V history written position by
// position). qkv row = [q heads | k heads | v heads]; pairs (j, j + hd/2), read
// from columns j and j + hd/2 of the head, or (PAIRED) 2j and 2j + 1.
template <bool PAIRED>
__global__ void __launch_bounds__(kRowThreads)
    k_rope_kv(const float* __restrict__ qkv, int start_pos, int H, int Hkv, int hd, const float2* __restrict__ table,
              float* __restrict__ q_out, float* __restrict__ k_cache, float* __restrict__ v_cache) {
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  const int i = blockIdx.x;
  const int pos = start_pos + i;
  const int half = hd / 2;
  const int ld = (H + 2 * Hkv) * hd;
  const float* row = qkv + (size_t)i * ld;
  const float2* tab = table + (size_t)pos * half;
  const int n_rot = (H + Hkv) * half;
  for (int e = threadIdx.x; e < n_rot; e += kRowThreads) {
    const int head = e / half, j = e % half;
    const float2 cs = tab[j];
    const float a = PAIRED ? row[head * hd + 2 * j] : row[head * hd + j];
    const float b = PAIRED ? row[head * hd + 2 * j + 1] : row[head * hd + j + half];
    const float2 r2 = ppdev::rope_rot(a, b, cs);
    const float ra = r2.x, rb = r2.y;
    if (head < H) {
      float* dst = q_out + ((size_t)i * H + head) * hd;
      dst[j] = ra;
      dst[j + half] = rb;
    } else {
      float* dst = k_cache + ((size_t)pos * Hkv + (head - H)) * hd;
      dst[j] = ra;
      dst[j + half] = rb;
    }
  }
  const float* vrow = row + (size_t)(H + Hkv) * hd;
  float* vdst = v_cache + (size_t)pos * Hkv * hd;
  for (int e = threadIdx.x; e < Hkv * hd; e += kRowThreads) vdst[e] = vrow[e];
}

// Output projection of the last position ("Single-pass prefill": logits for
// the last position only). Each warp takes kLmRows vocabulary rows at a time and
// walks their k range together, so the loads of all of them are in flight at
// once; the int32 dot products are exact, so neither the lane split nor the
// row grouping changes a result.
constexpr int kLmRows = 4;

__global__ void __launch_bounds__(kRowThreads)
    k_lm_head(const int8_t* __restrict__ q8, const float* __restrict__ a_scale, const int8_t* __restrict__ w,
              const float* __restrict__ ws, int vocab, int dim, float* __restrict__ logits) {
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  extern __shared__ int4 qs[];
  const int n16 = dim / 16;
  for (int c = threadIdx.x; c < n16; c += kRowThreads) qs[c] = reinterpret_cast<const int4*>(q8)[c];
  __syncthreads();
  const float as = a_scale[0];
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * kRowThreads + threadIdx.x) >> 5;
  const int n_warps = (gridDim.x * kRowThreads) >> 5;
  const int4* w4 = reinterpret_cast<const int4*>(w);
  for (int v0 = warp * kLmRows; v0 < vocab; v0 += n_warps * kLmRows) {
    int acc[kLmRows];
    const int4* wr[kLmRows];
#pragma unroll
    for (int r = 0; r < kLmRows; ++r) {
      acc[r] = 0;
      wr[r] = w4 + (size_t)min(v0 + r, vocab - 1) * n16;  // rows past the end repeat the last; never stored
    }
#pragma unroll 2
    for (int c = lane; c < n16; c += 32) {
      const int4 b = qs[c];
      int4 a[kLmRows];
#pragma unroll
      for (int r = 0; r < kLmRows; ++r) a[r] = __ldg(wr[r] + c);
#pragma unroll
      for (int r = 0; r < kLmRows; ++r) {
        acc[r] = __dp4a(a[r].x, b.x, acc[r]);
        acc[r] = __dp4a(a[r].y, b.y, acc[r]);
        acc[r] = __dp4a(a[r].z, b.z, acc[r]);
        acc[r] = __dp4a(a[r].w, b.w, acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kLmRows; ++r) {
      int v = acc[r];
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && v0 + r < vocab) logits[v0 + r] = ppdev::dequant(v, ws[v0 + r], as);
    }
  }
}

// int8 codes widened to fp16 (every integer in [-128, 127] is an fp16 value):
// the tcgen05 engine's activation operand for codes that arrive as int8.
__global__ void k_widen_i8(const int8_t* __restrict__ a, long long n, __half* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = __int2half_rn(a[i]);
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device(cache, [] {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
  });
}

}  // namespace

cudaError_t launch_embed(const int32_t* tok, int n, const float* emb, int vocab, int dim, float* x, int* status,
                         cudaStream_t s, bool pdl) {
  return launch_pdl_if(pdl, k_embed, dim3(n), dim3(kRowThreads), 0, s, tok, emb, vocab, dim, x, status);
}

cudaError_t launch_norm_quant(const float* x, int ldx, const float* g, int rows, int k, float eps, float* y,
                              int8_t* q8, __half* q16, float* a_scale, cudaStream_t s, bool pdl) {
  const int nv = (k / 4 + kRowThreads - 1) / kRowThreads;  // float4 per thread
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kern) {
    e = launch_pdl_if(pdl, kern, dim3(rows), dim3(kRowThreads), 0, s, x, ldx, g, k, eps, y, q8, q16, a_scale);
  };
  if (g) {
    if (nv <= 4) go(k_norm_quant<true, 4>);
    else if (nv <= 16) go(k_norm_quant<true, 16>);
    else go(k_norm_quant<true, 0>);
  } else {
    if (nv <= 4) go(k_norm_quant<false, 4>);
    else if (nv <= 16) go(k_norm_quant<false, 16>);
    else go(k_norm_quant<false, 0>);
  }
  return e;
}

cudaError_t launch_widen_i8(const int8_t* a, long long n, __half* out, cudaStream_t s) {
  k_widen_i8<<<sm_count() * 8, 256, 0, s>>>(a, n, out);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(int max_pos, int hd, float theta, float* table, cudaStream_t s) {
  k_rope_table<<<sm_count() * 4, 256, 0, s>>>(max_pos, hd, (double)theta, reinterpret_cast<float2*>(table));
  return cudaGetLastError();
}

cudaError_t launch_rope_kv(const float* qkv, int rows, int start_pos, int H, int Hkv, int hd, const float* table,
                           float* q_out, float* k_cache, float* v_cache, cudaStream_t s, bool paired, bool pdl) {
  return launch_pdl_if(pdl, paired ? k_rope_kv<true> : k_rope_kv<false>, dim3(rows), dim3(kRowThreads), 0, s, qkv, start_pos,
                    H, Hkv, hd, reinterpret_cast<const float2*>(table), q_out, k_cache, v_cache);
}

cudaError_t launch_lm_head(const int8_t* q8, const float* a_scale, const int8_t* w, const float* ws, int vocab,
                           int dim, float* logits, cudaStream_t s, bool pdl) {
  const int blocks = sm_count() * 4;
  return launch_pdl_if(pdl, k_lm_head, dim3(blocks), dim3(kRowThreads), (size_t)dim, s, q8, a_scale, w, ws, vocab, dim, logits);
}

}  // namespace pp
