// int8 x int8 -> int32 GEMM on warp-level mma.sync (m16n8k32, s8), the exact
// baseline engine of the projections ("Batched Prefill", "The Solution": one
// weight row dotted against many token columns, activations quantised once
// per chunk). acc[t][r] = sum_i a[t][i] * w[r][i] is exact in int32, so any
// tiling gives the same integers as the per-token GEMV.
//
// Tile 128 tokens x 128 weight rows x 64 k, 8 warps (2 x 4, 64 x 32 each),
// 4-stage cp.async pipeline, XOR-swizzled 64-byte smem rows read by
// ldmatrix. The epilogue applies (float(acc) * w_scale) * a_scale and,
// optionally, the residual add or SwiGLU of interleaved gate/up rows.
#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int STAGE_BYTES = (BM + BN) * BK;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES;

// Row r, 16-byte chunk c (0..3) of a 64-byte row, swizzled so that the 8 rows
// one ldmatrix phase touches land in 8 distinct bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

template <int EPI>
__global__ void __launch_bounds__(THREADS) k_gemm_mma(const int8_t* __restrict__ A, const int8_t* __restrict__ W,
                                                      const float* __restrict__ ws, const float* __restrict__ as,
                                                      int M, int N, int K, float* __restrict__ out, int ldo,
                                                      int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;
  const int ktiles = K / BK;

  int32_t acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

  auto load_stage = [&](int stage, int kt) {
    uint8_t* sa = smem + stage * STAGE_BYTES;
    uint8_t* sw = sa + BM * BK;
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + i * THREADS;
      const int row = c >> 2, ch = c & 3;
      const int gm = m0 + row, gn = n0 + row;
      ppdev::cp_async16(sa + swz(row, ch), A + (size_t)(gm < M ? gm : M - 1) * K + k0 + ch * 16, gm < M ? 16 : 0);
      ppdev::cp_async16(sw + swz(row, ch), W + (size_t)(gn < N ? gn : N - 1) * K + k0 + ch * 16, gn < N ? 16 : 0);
    }
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    ppdev::cp_async_commit();
  }

  for (int kt = 0; kt < ktiles; ++kt) {
    ppdev::cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nk = kt + STAGES - 1;
      if (nk < ktiles) load_stage(nk % STAGES, nk);
      ppdev::cp_async_commit();
    }
    const uint8_t* sa = smem + (kt % STAGES) * STAGE_BYTES;
    const uint8_t* sw = sa + BM * BK;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int mf = 0; mf < 4; ++mf) {
        const int row = wm * 64 + mf * 16 + (lane & 15);
        ppdev::ldmatrix_x4(af[mf], sa + swz(row, ks * 2 + (lane >> 4)));
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int nrow = wn * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        uint32_t r[4];
        ppdev::ldmatrix_x4(r, sw + swz(nrow, ks * 2 + ((lane >> 3) & 1)));
        bf[np * 2][0] = r[0];
        bf[np * 2][1] = r[1];
        bf[np * 2 + 1][0] = r[2];
        bf[np * 2 + 1][1] = r[3];
      }
#pragma unroll
      for (int mf = 0; mf < 4; ++mf)
#pragma unroll
        for (int nf = 0; nf < 4; ++nf) ppdev::mma_s8_16832(acc[mf][nf], af[mf], bf[nf]);
    }
  }
  ppdev::cp_async_wait<0>();

  // ---- epilogue
  const int group = lane >> 2, tig = lane & 3;
  const int wcol = n0 + wn * 32;
  if (wcol >= N) return;
#pragma unroll
  for (int mf = 0; mf < 4; ++mf) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = m0 + wm * 64 + mf * 16 + group + half * 8;
      if (row >= M) continue;
      if (EPI == EPI_ACC) {
#pragma unroll
        for (int nf = 0; nf < 4; ++nf) {
          const int col = wcol + nf * 8 + 2 * tig;
          *reinterpret_cast<int2*>(acc_out + (size_t)row * N + col) =
              make_int2(acc[mf][nf][half * 2], acc[mf][nf][half * 2 + 1]);
        }
        continue;
      }
      const float a_s = as[row];
      if (EPI == EPI_SWIGLU) {
        // warp columns [wcol, wcol+32) = 16 gate rows then 16 up rows of one block
#pragma unroll
        for (int f = 0; f < 2; ++f) {
          const int cg = wcol + f * 8 + 2 * tig;
          const float g0 = ppdev::dequant(acc[mf][f][half * 2], ws[cg], a_s);
          const float g1 = ppdev::dequant(acc[mf][f][half * 2 + 1], ws[cg + 1], a_s);
          const float u0 = ppdev::dequant(acc[mf][f + 2][half * 2], ws[cg + 16], a_s);
          const float u1 = ppdev::dequant(acc[mf][f + 2][half * 2 + 1], ws[cg + 17], a_s);
          const int hc = wcol / 2 + f * 8 + 2 * tig;
          *reinterpret_cast<float2*>(out + (size_t)row * ldo + hc) =
              make_float2(ppdev::silu_mul(g0, u0), ppdev::silu_mul(g1, u1));
        }
      } else {
#pragma unroll
        for (int nf = 0; nf < 4; ++nf) {
          const int col = wcol + nf * 8 + 2 * tig;
          float v0 = ppdev::dequant(acc[mf][nf][half * 2], ws[col], a_s);
          float v1 = ppdev::dequant(acc[mf][nf][half * 2 + 1], ws[col + 1], a_s);
          float2* dst = reinterpret_cast<float2*>(out + (size_t)row * ldo + col);
          if (EPI == EPI_RESID) {
            const float2 r = *dst;
            v0 = __fadd_rn(r.x, v0);
            v1 = __fadd_rn(r.y, v1);
          }
          *dst = make_float2(v0, v1);
        }
      }
    }
  }
}

template <int EPI>
cudaError_t launch_t(const int8_t* a8, const int8_t* w, const float* ws, const float* as, int m, int n, int k,
                     float* out, int ldo, int32_t* acc, cudaStream_t s) {
  static std::atomic<uint64_t> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(k_gemm_mma<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  dim3 grid((n + BN - 1) / BN, (m + BM - 1) / BM);
  k_gemm_mma<EPI><<<grid, THREADS, SMEM_BYTES, s>>>(a8, w, ws, as, m, n, k, out, ldo, acc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mma(int epi, const int8_t* a8, const int8_t* w, const float* ws, const float* as, int m,
                            int n, int k, float* out, int ldo, int32_t* acc, cudaStream_t s) {
  switch (epi) {
    case EPI_STORE: return launch_t<EPI_STORE>(a8, w, ws, as, m, n, k, out, ldo, acc, s);
    case EPI_RESID: return launch_t<EPI_RESID>(a8, w, ws, as, m, n, k, out, ldo, acc, s);
    case EPI_SWIGLU: return launch_t<EPI_SWIGLU>(a8, w, ws, as, m, n, k, out, ldo, acc, s);
    case EPI_ACC: return launch_t<EPI_ACC>(a8, w, ws, as, m, n, k, out, ldo, acc, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pp
