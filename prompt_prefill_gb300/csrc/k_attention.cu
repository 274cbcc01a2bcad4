// Causal chunk attention over the K/V cache, f32 on CUDA cores.
//
// "Single-pass prefill": position i attends over kv[layer][0..i], which is
// already written because K/V rows of the chunk are written before this
// kernel runs (each row depends only on its own position). "Batched Prefill",
// "What Stays Sequential": attention is sequential in positions; here every
// position of the chunk is one independent query row, which is equivalent.
//
// Work split. A query tile is 64 rows (64/G positions x the G query heads
// that share a KV head). Its keys are cut into ranges of kAttnRange keys at
// fixed absolute positions (0, 512, 1024, ...), and one CTA runs one (tile,
// KV head, range) item, heaviest items first, so the grid fills every SM
// evenly whatever the chunk's position. Within an item the key axis streams
// through shared memory in blocks of 64 keys; per row: online softmax in
// base 2 (q pre-scaled by log2(e)/sqrt(hd)), warp-shuffle max/sum over the 8
// lanes that hold the row, then O += P V. A tile whose keys fit one range
// writes o directly; otherwise every item writes its (O, m, l) state and a
// second kernel combines the ranges of each row in range order.
//
// Chunk invariance. The ranges, the blocks within a range and the order of
// every reduction depend only on a row's absolute position: a block or a
// range past the row's position is fully masked and leaves its state (or the
// merged result) bit-for-bit unchanged, so a row's result does not depend on
// the chunk it was computed in.
#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int ROWS = 64;      // query rows per CTA
constexpr int KB = 64;        // keys per block
constexpr int NB = KB / 8;    // keys per thread in a block (tx + 8b)
constexpr int CTAS_PER_SM = 2;
constexpr int THREADS = 128;  // 16 row groups (ty) x 8 lanes (tx)
constexpr int PS = 68;        // padded stride of the P tile, [key][4 ty + a]
static_assert(kAttnRange % KB == 0, "a key range is a whole number of key blocks");
// A row's reference maximum is raised only when a block's maximum exceeds it
// by more than this (base-2 units), so unnormalised p stays below 2^kLazy.
constexpr float kLazy = 8.f;

// 2^x by the hardware approximation (relative error ~2^-22; 2^-inf = 0, and
// results below 2^-126 flush to 0, which no sum here can notice).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// XOR swizzle of 16-byte chunks within a row of the Q and K tiles: rows r and
// r' with r = r' (mod 8) never share a bank group when read at the same d.
template <int HD>
__device__ __forceinline__ int swz(int r, int d) {
  return r * HD + ((((d >> 2) ^ (r & 7))) << 2) + (d & 3);
}

struct Tile {
  int tile, kvh, i0, pmax, nr;  // query tile, KV head, first row, last position, number of key ranges
};

__device__ __forceinline__ Tile tile_of(int j, int n_tiles, int Hkv, int bq, int C, int start_pos) {
  Tile t;
  t.tile = n_tiles - 1 - j / Hkv;  // later positions (more keys) first
  t.kvh = j % Hkv;
  t.i0 = t.tile * bq;
  t.pmax = start_pos + min(t.i0 + bq, C) - 1;
  t.nr = t.pmax / kAttnRange + 1;
  return t;
}

template <int HD>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    k_attention(const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc, int C,
                int start_pos, int H, int Hkv, float* __restrict__ o, float qscale, float* __restrict__ part,
                int n_ranges) {
  extern __shared__ __align__(16) float sm[];
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  float* Qs = sm;              // [ROWS][HD] swizzled
  float* Ks = Qs + ROWS * HD;  // [KB][HD] swizzled
  float* Vs = Ks + KB * HD;    // [KB][HD]
  float* Ps = Vs + KB * HD;    // [KB][PS]

  const int G = H / Hkv;
  const int bq = ROWS / G;  // positions per tile
  const int n_tiles = (C + bq - 1) / bq;
  const int per_range = n_tiles * Hkv;
  const int r = blockIdx.x / per_range;
  const Tile T = tile_of(blockIdx.x % per_range, n_tiles, Hkv, bq, C, start_pos);
  if (r >= T.nr) return;  // no key of this range is visible to the tile
  const int kvh = T.kvh, i0 = T.i0, pmax = T.pmax;
  const int kb_begin = r * (kAttnRange / KB);
  const int kb_end = min(pmax, (r + 1) * kAttnRange - 1) / KB + 1;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;

  constexpr int C4 = HD / 4;
  // K/V tiles stream through shared memory with cp.async: K of block kb+1
  // loads while softmax and P V of block kb run, V of block kb+1 while S of
  // block kb+1 runs. Two CTA barriers per block: before each, every thread
  // waits for its own copies in flight (V of the block before the first, K of
  // the next block before the second), so each barrier both frees a buffer
  // and publishes the copy that lands in the other. P is private to a warp
  // (a thread reads only the rows of its own ty), so it needs only __syncwarp.
  // Keys past the tile's last position are zero-filled.
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
  load_tile(Ks, kc, kb_begin * KB, true);
  load_tile(Vs, vc, kb_begin * KB, false);

  // Query tile (issued after the first K/V copies, so the latencies overlap;
  // row rr = position-in-tile * G + head-in-group).
#pragma unroll 8
  for (int e = tid; e < ROWS * C4; e += THREADS) {
    const int rr = e / C4, c = e % C4;
    int i = i0 + rr / G;
    if (i > C - 1) i = C - 1;  // padding rows recompute the last position; never stored
    const int h = kvh * G + rr % G;
    float4 v = *reinterpret_cast<const float4*>(q + ((size_t)i * H + h) * HD + 4 * c);
    v.x *= qscale; v.y *= qscale; v.z *= qscale; v.w *= qscale;
    *reinterpret_cast<float4*>(&Qs[swz<HD>(rr, 4 * c)]) = v;
  }

  // This thread's rows: ty + 16a; its keys in a block: tx + 8b; its dims: 4tx + 32i + e.
  int pos[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    int i = i0 + (ty + 16 * a) / G;
    if (i > C - 1) i = C - 1;
    pos[a] = start_pos + i;
  }
  const int pos_lo = start_pos + i0;  // the tile's first position: no key below it is masked

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

  ppdev::cp_async_wait<1>();  // K of the first block (V may still be in flight)
  __syncthreads();

  for (int kb = kb_begin; kb < kb_end; ++kb) {
    const int key0 = kb * KB;
    const bool more = kb + 1 < kb_end;

    // S = Q K^T for rows ty+16a, keys tx+8b. Packed f32 FMA over pairs of d:
    // Sp[a][b].x sums the even d, .y the odd d (in d order); S = .x + .y.
    float2 Sp[4][NB];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b) Sp[a][b] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int d = 0; d < HD; d += 4) {
      float4 qv[4], kv[NB];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = *reinterpret_cast<const float4*>(&Qs[swz<HD>(ty + 16 * a, d)]);
#pragma unroll
      for (int b = 0; b < NB; ++b) kv[b] = *reinterpret_cast<const float4*>(&Ks[swz<HD>(tx + 8 * b, d)]);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b)
          Sp[a][b] = __ffma2_rn(make_float2(qv[a].x, qv[a].y), make_float2(kv[b].x, kv[b].y), Sp[a][b]);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b)
          Sp[a][b] = __ffma2_rn(make_float2(qv[a].z, qv[a].w), make_float2(kv[b].z, kv[b].w), Sp[a][b]);
    }
    float S[4][NB];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b) S[a][b] = Sp[a][b].x + Sp[a][b].y;
    ppdev::cp_async_wait<0>();  // V of this block
    __syncthreads();            // every warp is done with Ks; V of this block visible
    if (more) load_tile(Ks, kc, key0 + KB, true);

    // Causal mask (only in a block that crosses the tile's first position),
    // then online softmax in base 2. The reference maximum m of a row moves
    // only when a block's maximum exceeds it by more than kLazy, so p stays
    // below 2^kLazy and the O rescale is skipped by every warp whose rows all
    // kept their m. A row that has seen no key of this range yet (m = -inf)
    // keeps m = -inf, l = 0, O = 0 through masked blocks.
    if (key0 + KB - 1 > pos_lo) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (key0 + tx + 8 * b > pos[a]) S[a][b] = -INFINITY;
    }
    float alpha[4];
    bool rescale = false;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float mb = S[a][0];
#pragma unroll
      for (int b = 1; b < NB; ++b) mb = fmaxf(mb, S[a][b]);
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      alpha[a] = 1.f;
      if (mb > m[a] + kLazy) {  // false for mb = -inf; true for the first finite block of a row
        alpha[a] = ex2(m[a] - mb);
        m[a] = mb;
        rescale = true;
      }
      const float mref = (m[a] == -INFINITY) ? 0.f : m[a];
      float ls = 0.f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float p = ex2(S[a][b] - mref);
        ls += p;
        S[a][b] = p;
      }
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      ls += __shfl_xor_sync(0xffffffffu, ls, 4);
      l[a] = fmaf(l[a], alpha[a], ls);
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int i = 0; i < ND; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) O[a][i][e] *= alpha[a];
    }
    // P -> smem, the thread's 4 rows of one key as one 16-byte store
#pragma unroll
    for (int b = 0; b < NB; ++b)
      *reinterpret_cast<float4*>(&Ps[(tx + 8 * b) * PS + 4 * ty]) = make_float4(S[0][b], S[1][b], S[2][b], S[3][b]);
    __syncwarp();  // the warp's P rows are written

    // O += P V, keys in order (unrolled 32 deep: measured 1.7% faster than 8).
#pragma unroll 32
    for (int j = 0; j < KB; ++j) {
      const float4 p4 = *reinterpret_cast<const float4*>(&Ps[j * PS + 4 * ty]);
      const float p[4] = {p4.x, p4.y, p4.z, p4.w};
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
    ppdev::cp_async_wait<0>();  // K of the next block
    __syncthreads();            // every warp is done with Vs; K of the next block visible
    if (more) load_tile(Vs, vc, key0 + KB, false);
  }
  ppdev::cp_async_wait<0>();

  if (T.nr == 1) {
    // o[i][h][:] = O / l
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int rr = ty + 16 * a;
      const int i = i0 + rr / G;
      if (i >= C) continue;
      const int h = kvh * G + rr % G;
      const float inv_l = 1.0f / l[a];
      float* dst = o + ((size_t)i * H + h) * HD;
#pragma unroll
      for (int ii = 0; ii < ND; ++ii)
        *reinterpret_cast<float4*>(dst + 4 * tx + 32 * ii) =
            make_float4(O[a][ii][0] * inv_l, O[a][ii][1] * inv_l, O[a][ii][2] * inv_l, O[a][ii][3] * inv_l);
    }
    return;
  }
  // This range's state: O (not normalised) [ROWS][HD], then (m, l) [ROWS].
  float* po = part + ((size_t)(T.tile * Hkv + kvh) * n_ranges + r) * ROWS * (HD + 2);
  float* pml = po + ROWS * HD;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int rr = ty + 16 * a;
#pragma unroll
    for (int ii = 0; ii < ND; ++ii)
      *reinterpret_cast<float4*>(po + rr * HD + 4 * tx + 32 * ii) =
          make_float4(O[a][ii][0], O[a][ii][1], O[a][ii][2], O[a][ii][3]);
    if (tx == 0) *reinterpret_cast<float2*>(pml + 2 * rr) = make_float2(m[a], l[a]);
  }
}

// Combine the ranges of every tile that has more than one, in range order,
// one thread per (row, 4 dims): m = max_r m_r, O = sum_r O_r 2^(m_r - m),
// l = sum_r l_r 2^(m_r - m), o = O / l. A range with m_r = -inf (no key of it
// is visible to the row) is skipped, so a row that sees one range gets
// O_0 * 1 / l_0 * 1: the same bits as the single-range path.
template <int HD>
__global__ void __launch_bounds__(256)
    k_attention_merge(int C, int start_pos, int H, int Hkv, float* __restrict__ o, const float* __restrict__ part,
                      int n_ranges) {
  ppdev::pdl_trigger();
  ppdev::pdl_wait();
  constexpr int F4 = HD / 4;
  constexpr int CTAS_PER_TILE = ROWS * F4 / 256;
  const int G = H / Hkv;
  const int bq = ROWS / G;
  const int n_tiles = (C + bq - 1) / bq;
  const Tile T = tile_of(blockIdx.x / CTAS_PER_TILE, n_tiles, Hkv, bq, C, start_pos);
  if (T.nr == 1) return;
  const int e = (blockIdx.x % CTAS_PER_TILE) * 256 + threadIdx.x;
  const int rr = e / F4, d4 = e % F4;
  const int i = T.i0 + rr / G;
  if (i >= C) return;
  const size_t stride = (size_t)ROWS * (HD + 2);
  const float* base = part + (size_t)(T.tile * Hkv + T.kvh) * n_ranges * stride;
  float mx = -INFINITY;
#pragma unroll 8
  for (int r = 0; r < T.nr; ++r) mx = fmaxf(mx, base[r * stride + ROWS * HD + 2 * rr]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  bool first = true;
#pragma unroll 8
  for (int r = 0; r < T.nr; ++r) {
    const float2 ml = *reinterpret_cast<const float2*>(base + r * stride + ROWS * HD + 2 * rr);
    if (ml.x == -INFINITY) continue;
    const float s = exp2f(ml.x - mx);
    const float4 v = *reinterpret_cast<const float4*>(base + r * stride + rr * HD + 4 * d4);
    if (first) {
      acc = make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
      L = ml.y * s;
      first = false;
    } else {
      acc = make_float4(fmaf(v.x, s, acc.x), fmaf(v.y, s, acc.y), fmaf(v.z, s, acc.z), fmaf(v.w, s, acc.w));
      L = fmaf(ml.y, s, L);
    }
  }
  const float inv_l = 1.0f / L;
  const int h = T.kvh * G + rr % G;
  *reinterpret_cast<float4*>(o + ((size_t)i * H + h) * HD + 4 * d4) =
      make_float4(acc.x * inv_l, acc.y * inv_l, acc.z * inv_l, acc.w * inv_l);
}

template <int HD>
cudaError_t launch_t(const float* q, const float* kc, const float* vc, int rows, int start_pos, int H, int Hkv,
                     float* o, float* part, size_t part_bytes, cudaStream_t s, bool pdl) {
  constexpr int smem = (ROWS * HD + 2 * KB * HD + KB * PS) * (int)sizeof(float);
  static std::atomic<uint64_t> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(k_attention<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  const int G = H / Hkv;
  const int bq = ROWS / G;
  const int n_tiles = (rows + bq - 1) / bq;
  const int n_ranges = (start_pos + rows - 1) / kAttnRange + 1;
  if (n_ranges > 1 && (!part || part_bytes < attention_workspace_bytes(rows, start_pos, H, Hkv, HD)))
    return cudaErrorInvalidValue;
  const float qscale = (float)(1.4426950408889634 / sqrt((double)HD));
  e = launch_pdl_if(pdl, k_attention<HD>, dim3(n_tiles * Hkv * n_ranges), dim3(THREADS), (size_t)smem, s, q, kc, vc,
                    rows, start_pos, H, Hkv, o, qscale, part, n_ranges);
  if (e == cudaSuccess && n_ranges > 1)
    e = launch_pdl(k_attention_merge<HD>, dim3(n_tiles * Hkv * (ROWS * HD / 4 / 256)), dim3(256), 0, s, rows,
                   start_pos, H, Hkv, o, (const float*)part, n_ranges);
  return e;
}

}  // namespace

size_t attention_workspace_bytes(int rows, int start_pos, int H, int Hkv, int hd) {
  const int bq = ROWS / (H / Hkv);
  const size_t n_tiles = (size_t)(rows + bq - 1) / bq;
  const size_t n_ranges = (size_t)(start_pos + rows - 1) / kAttnRange + 1;
  if (n_ranges == 1) return 0;
  return n_tiles * Hkv * n_ranges * ROWS * (hd + 2) * sizeof(float);
}

cudaError_t launch_attention(const float* q, const float* kc, const float* vc, int rows, int start_pos, int H,
                             int Hkv, int hd, float* o, float* part, size_t part_bytes, cudaStream_t s, bool pdl) {
  if (hd == 64) return launch_t<64>(q, kc, vc, rows, start_pos, H, Hkv, o, part, part_bytes, s, pdl);
  if (hd == 128) return launch_t<128>(q, kc, vc, rows, start_pos, H, Hkv, o, part, part_bytes, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace pp
