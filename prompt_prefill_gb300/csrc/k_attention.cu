// Causal chunk attention over the K/V cache, f32 on CUDA cores.
//
// "Single-pass prefill": position i attends over kv[layer][0..i], which is
// already written because K/V rows of the chunk are written before this
// kernel runs (each row depends only on its own position). "Batched Prefill",
// "What Stays Sequential": attention is sequential in positions; here every
// position of the chunk is one independent query row, which is equivalent.
//
// One CTA = one KV head x a tile of 64 query rows (64/G positions x the G
// query heads that share the KV head), streaming the key axis in blocks of
// 64 keys aligned to absolute positions. Per row: online softmax in base 2
// (q pre-scaled by log2(e)/sqrt(hd)), warp-shuffle max/sum over the 8 lanes
// that hold the row, then O += P V. Blocks are walked in the same order for
// every query; a block past a row's own position is fully masked, which
// leaves its state bit-for-bit unchanged (alpha = 1, p = 0). A row's result
// therefore depends only on its absolute position and the cache, not on the
// chunk it was computed in.
#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int ROWS = 64;     // query rows per CTA
constexpr int KB = 64;       // keys per block
constexpr int THREADS = 128; // 16 row groups (ty) x 8 lanes (tx)
constexpr int PS = 68;       // padded stride of the P tile

// XOR swizzle of 16-byte chunks within a row of the Q and K tiles: rows r and
// r' with r = r' (mod 8) never share a bank group when read at the same d.
template <int HD>
__device__ __forceinline__ int swz(int r, int d) {
  return r * HD + ((((d >> 2) ^ (r & 7))) << 2) + (d & 3);
}

template <int HD>
__global__ void __launch_bounds__(THREADS, 2)
    k_attention(const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc, int C,
                int start_pos, int H, int Hkv, float* __restrict__ o, float qscale) {
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                  // [ROWS][HD] swizzled
  float* Ks = Qs + ROWS * HD;      // [KB][HD] swizzled
  float* Vs = Ks + KB * HD;        // [KB][HD]
  float* Ps = Vs + KB * HD;        // [KB][PS]

  const int G = H / Hkv;
  const int bq = ROWS / G;  // positions per tile
  const int kvh = blockIdx.y;
  const int i0 = blockIdx.x * bq;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;

  // Load the query tile (row r = position-in-tile * G + head-in-group).
  constexpr int C4 = HD / 4;
  for (int e = tid; e < ROWS * C4; e += THREADS) {
    const int r = e / C4, c = e % C4;
    int i = i0 + r / G;
    if (i > C - 1) i = C - 1;  // padding rows recompute the last position; never stored
    const int h = kvh * G + r % G;
    float4 v = *reinterpret_cast<const float4*>(q + ((size_t)i * H + h) * HD + 4 * c);
    v.x *= qscale; v.y *= qscale; v.z *= qscale; v.w *= qscale;
    *reinterpret_cast<float4*>(&Qs[swz<HD>(r, 4 * c)]) = v;
  }

  // This thread's rows: ty + 16a; its keys in a block: tx + 8b; its dims: 4tx + 32i + e.
  int pos[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    int i = i0 + (ty + 16 * a) / G;
    if (i > C - 1) i = C - 1;
    pos[a] = start_pos + i;
  }
  const int last_i = min(i0 + bq, C) - 1;
  const int pmax = start_pos + last_i;
  const int nblocks = pmax / KB + 1;

  constexpr int ND = HD / 32;  // float4 groups of dims per thread
  float O[4][ND][4];
  float m[4], l[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int i = 0; i < ND; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[a][i][e] = 0.f;
  }

  // K/V tiles stream through shared memory with cp.async: K of block kb+1
  // loads while P V of block kb runs, V of block kb+1 while S of block kb+1
  // runs. Keys past the tile's last position are zero-filled.
  auto load_tile = [&](float* dst, const float* src, int key0, bool swizzle) {
    for (int e = tid; e < KB * C4; e += THREADS) {
      const int j = e / C4, c = e % C4;
      const int kp = key0 + j;
      const bool ok = kp <= pmax;
      const float* g = src + ((size_t)(ok ? kp : 0) * Hkv + kvh) * HD + 4 * c;
      float* d = swizzle ? &dst[swz<HD>(j, 4 * c)] : &dst[j * HD + 4 * c];
      ppdev::cp_async16(d, g, ok ? 16 : 0);
    }
    ppdev::cp_async_commit();
  };
  load_tile(Ks, kc, 0, true);
  load_tile(Vs, vc, 0, false);
  ppdev::cp_async_wait<1>();  // K of block 0
  __syncthreads();

  for (int kb = 0; kb < nblocks; ++kb) {
    const int key0 = kb * KB;
    const bool more = kb + 1 < nblocks;

    // S = Q K^T for rows ty+16a, keys tx+8b, in d order.
    float S[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) S[a][b] = 0.f;
#pragma unroll 4
    for (int d = 0; d < HD; d += 4) {
      float4 qv[4], kv[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = *reinterpret_cast<const float4*>(&Qs[swz<HD>(ty + 16 * a, d)]);
#pragma unroll
      for (int b = 0; b < 8; ++b) kv[b] = *reinterpret_cast<const float4*>(&Ks[swz<HD>(tx + 8 * b, d)]);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          S[a][b] = fmaf(qv[a].x, kv[b].x, S[a][b]);
          S[a][b] = fmaf(qv[a].y, kv[b].y, S[a][b]);
          S[a][b] = fmaf(qv[a].z, kv[b].z, S[a][b]);
          S[a][b] = fmaf(qv[a].w, kv[b].w, S[a][b]);
        }
    }
    __syncthreads();  // every warp is done with Ks
    if (more) load_tile(Ks, kc, key0 + KB, true);
    else ppdev::cp_async_commit();

    // Causal mask, online softmax (base 2), P -> smem.
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float mb = -INFINITY;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (key0 + tx + 8 * b > pos[a]) S[a][b] = -INFINITY;
        mb = fmaxf(mb, S[a][b]);
      }
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      const float mn = fmaxf(m[a], mb);
      const float alpha = (mn == m[a]) ? 1.f : exp2f(m[a] - mn);
      float ls = 0.f;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const float p = exp2f(S[a][b] - mn);
        ls += p;
        Ps[(tx + 8 * b) * PS + ty + 16 * a] = p;
      }
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      ls += __shfl_xor_sync(0xffffffffu, ls, 4);
      l[a] = l[a] * alpha + ls;
      m[a] = mn;
#pragma unroll
      for (int i = 0; i < ND; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[a][i][e] *= alpha;
    }
    ppdev::cp_async_wait<1>();  // V of this block (the K prefetch may still be in flight)
    __syncthreads();

    // O += P V, keys in order.
#pragma unroll 4
    for (int j = 0; j < KB; ++j) {
      float p[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) p[a] = Ps[j * PS + ty + 16 * a];
#pragma unroll
      for (int i = 0; i < ND; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(&Vs[j * HD + 4 * tx + 32 * i]);
        const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          // packed f32 FMA: two independent round-to-nearest FMAs per instruction
          const float2 pp = make_float2(p[a], p[a]);
          float2 o01 = make_float2(O[a][i][0], O[a][i][1]), o23 = make_float2(O[a][i][2], O[a][i][3]);
          o01 = __ffma2_rn(pp, v01, o01);
          o23 = __ffma2_rn(pp, v23, o23);
          O[a][i][0] = o01.x;
          O[a][i][1] = o01.y;
          O[a][i][2] = o23.x;
          O[a][i][3] = o23.y;
        }
      }
    }
    __syncthreads();  // every warp is done with Vs and Ps
    if (more) load_tile(Vs, vc, key0 + KB, false);
    else ppdev::cp_async_commit();
    ppdev::cp_async_wait<1>();  // K of the next block
    __syncthreads();
  }
  ppdev::cp_async_wait<0>();

  // o[i][h][:] = O / l
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int r = ty + 16 * a;
    const int i = i0 + r / G;
    if (i >= C) continue;
    const int h = kvh * G + r % G;
    const float inv_l = 1.0f / l[a];
    float* dst = o + ((size_t)i * H + h) * HD;
#pragma unroll
    for (int ii = 0; ii < ND; ++ii)
      *reinterpret_cast<float4*>(dst + 4 * tx + 32 * ii) =
          make_float4(O[a][ii][0] * inv_l, O[a][ii][1] * inv_l, O[a][ii][2] * inv_l, O[a][ii][3] * inv_l);
  }
}

template <int HD>
cudaError_t launch_t(const float* q, const float* kc, const float* vc, int rows, int start_pos, int H, int Hkv,
                     float* o, cudaStream_t s) {
  constexpr int smem = (ROWS * HD + 2 * KB * HD + KB * PS) * (int)sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_attention<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int G = H / Hkv;
  const int bq = ROWS / G;
  dim3 grid((rows + bq - 1) / bq, Hkv);
  const float qscale = (float)(1.4426950408889634 / sqrt((double)HD));
  k_attention<HD><<<grid, THREADS, smem, s>>>(q, kc, vc, rows, start_pos, H, Hkv, o, qscale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const float* q, const float* kc, const float* vc, int rows, int start_pos, int H,
                             int Hkv, int hd, float* o, cudaStream_t s) {
  if (hd == 64) return launch_t<64>(q, kc, vc, rows, start_pos, H, Hkv, o, s);
  if (hd == 128) return launch_t<128>(q, kc, vc, rows, start_pos, H, Hkv, o, s);
  return cudaErrorInvalidValue;
}

}  // namespace pp
