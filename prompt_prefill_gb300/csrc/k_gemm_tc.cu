// Exact int8 x int8 -> int32 GEMM on the 5th-generation tensor cores.
//
// "Batched Prefill", "The Solution": each weight row is dotted against the
// whole chunk of token columns, with activations quantised once per chunk.
// sm_103a has no integer tcgen05 MMA kind, so the integer GEMM runs on
// tcgen05.mma.kind::f16 with operands that hold the int8 codes exactly:
//   - every integer in [-127, 127] is an fp16 value, and every product of two
//     such values (|a*w| <= 16129) is exact in the f32 accumulator;
//   - an f32 sum of such products is exact while every partial sum stays below
//     2^24 in magnitude, i.e. for up to floor(2^24 / 127^2) = 1040 products.
// The K axis is therefore cut into segments of at most 1024 (16 k-blocks of
// 64); each segment accumulates into its own f32 TMEM buffer, which drain
// warps read back, convert to int32 (exact) and add to int32 registers. The
// result equals the int32 dot product bit for bit.
//
// Layout: a CTA pair (cluster of 2, cta_group::2) computes a 256-token x
// BN-weight-row tile (BN = 256, 192 or 128, chosen per shape so that the
// tiles fill the 76 pairs); each CTA holds 128 token rows of A (fp16 codes,
// TMA, 128-byte swizzle) and BN/2 weight rows of B. Weights stay int8 in HBM:
// TMA brings int8 rows into shared memory and converter warps widen them to
// fp16 in the UMMA K-major 128-byte-swizzled layout (exponent-bias method:
// 0x6400 | (b ^ 0x80) is the fp16 number 1024 + 128 + b, minus 1152 gives b).
//
// Roles (16 warps): warp 0 issues TMA, warp 1 (leader CTA) issues the MMAs,
// warpgroup 1 only converts, warpgroups 2-3 only drain accumulators and run
// the epilogue (each thread holds BN/2 int32 running sums). Conversion never
// waits behind a drain or an epilogue, so the stages ahead of the tensor core
// stay filled. Persistent over tiles; two TMEM accumulators of BN columns
// alternate between segments. Every mbarrier wait is bounded: on expiry the
// kernel records a timeout in the status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int BM = 128;             // token rows per CTA (256 per pair)
constexpr int BK = 64;              // k per stage: 128 bytes of fp16
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int N_CONV_WARPS = 4;     // warpgroup 1: int8 -> fp16 conversion
constexpr int N_DRAIN_WARPS = 8;    // warpgroups 2-3: 2 per TMEM lane quarter, BN/2 accumulator columns each
constexpr int THREADS = 512;        // warpgroup 0: TMA, MMA, 2 idle
constexpr int CONV_WARP0 = 4;
constexpr int DRAIN_WARP0 = 8;
// Register split (setmaxnreg): launched at 128 per thread (16 x 32 x 128 = 65536 in the
// pool); warpgroup 0 drops to 40, the converters to 72 and the drain warpgroups rise to
// 200: 128 x 40 + 128 x 72 + 256 x 200 = 65536, and per SM sub-partition
// (40 + 72 + 200 + 200) x 32 = 16384.
constexpr int REGS_ROLE = 40, REGS_CONV = 72, REGS_DRAIN = 200;
constexpr int MAX_SEG_KB = 16;      // 16 x 64 = 1024 products per exact f32 segment
constexpr int MIN_SK_KB = 64;       // stream-K only when each cluster owns >= 64 k-blocks (measured: fixups
                                    // cost more than they recover at ~30-40 k-blocks per cluster)
constexpr int STAGE_BUDGET = 204 * 1024;  // shared memory for the pipeline stages
constexpr int EPI_LD = 20;  // floats per row of a drain warp's epilogue staging (16 + 4: conflict-free writes)

// Per-tile-width constants.
template <int BN>
struct Cfg {
  static constexpr int B_BYTES = (BN / 2) * BK * 2;  // converted weights of one CTA
  static constexpr int W_BYTES = (BN / 2) * BK;      // int8 weights of one CTA
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + W_BYTES;
  static constexpr int STAGES = STAGE_BUDGET / STAGE_BYTES;  // 5 (256), 6 (192), 7 (128)
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + 2 * BN * 4 /*w_scale*/ +
                                    N_DRAIN_WARPS * 32 * EPI_LD * 4 /*epilogue staging*/;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static constexpr int COLS = BN / 2;                 // accumulator columns per drain warp
  static_assert(B_BYTES % 1024 == 0 && W_BYTES % 1024 == 0, "stage buffers keep the 1024-byte swizzle alignment");
};

struct TcParams {
  int M, N, K;
  int seg_kb;
  int num_m_tiles, num_tiles;
  const float* ws;
  const float* as;
  float* out;
  int ldo;
  int32_t* acc_out;
  int* status;
  // stream-K: cluster c owns iterations [c*ipc, (c+1)*ipc) of the (tile, k-block)
  // space; partial tiles meet in `part` (int32, BM x BN per tile, slot and CTA) and the
  // last contributor, counted in `cnt` ([tile][cta], zero between launches), adds
  // the partial sums and runs the epilogue. ipc == 0: whole tiles round robin.
  int ipc;
  int max_slots;
  int32_t* part;
  int* cnt;
  TcRope rope;            // EPI_ROPE destinations
  long long wait_cycles;  // bound of every mbarrier wait (clock64 cycles)
  int hold_mma;           // test hook: the MMA issuer issues nothing, so every other role's wait runs out
  int early_w;            // the first stages' weight loads may precede griddepcontrol.wait
};

// The units (tile, k-block range) a cluster works on, in order.
struct Sched {
  int cluster, n_clusters, num_tiles, nkb, ipc, it0, it1;
  __device__ Sched(const TcParams& p, int c, int nc) : cluster(c), n_clusters(nc), num_tiles(p.num_tiles),
      nkb(p.K / BK), ipc(p.ipc) {
    const long long total = (long long)num_tiles * nkb;
    it0 = ipc ? (int)min((long long)c * ipc, total) : 0;
    it1 = ipc ? (int)min((long long)(c + 1) * ipc, total) : 0;
  }
  __device__ int units() const {
    if (!ipc) return num_tiles > cluster ? (num_tiles - cluster + n_clusters - 1) / n_clusters : 0;
    return it1 > it0 ? (it1 - 1) / nkb - it0 / nkb + 1 : 0;
  }
  __device__ void unit(int u, int& tile, int& kb0, int& kb1) const {
    if (!ipc) { tile = cluster + u * n_clusters; kb0 = 0; kb1 = nkb; return; }
    tile = it0 / nkb + u;
    kb0 = u == 0 ? it0 % nkb : 0;
    kb1 = tile == (it1 - 1) / nkb ? (it1 - 1) % nkb + 1 : nkb;
  }
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
// Arrive on the barrier at the same offset in CTA `rank` of the cluster, with
// the default (CTA-scope release) semantics. Callers that hand shared-memory
// data to the tensor core issue fence.proxy.async.shared::cta first. A
// cluster-scope release here costs a device-wide memory barrier per arrive
// and measured ~1.8x slower GEMMs; the data itself never leaves the writing
// CTA's shared memory, which the tensor core pair reads directly.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t a, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after ~2 s without the phase completing.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, long long limit) {
  if (mbar_try(a, parity)) return true;
  const long long end = clock64() + limit;
  while (!mbar_try(a, parity))
    if (clock64() > end) return false;
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// UMMA shared-memory descriptor: K-major operand in the 128-byte swizzle
// layout (8-row atoms of 1024 bytes stacked at 1024 bytes).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: f16 x f16 -> f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive once on barrier `a` in both CTAs of the pair when all prior MMAs of this thread complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t a) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(a),
      "h"((uint16_t)0x3)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Four int8 codes -> two f16x2 words holding the same integers.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;  // b + 128 as unsigned bytes
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));  // (1024 + 128 + b) - 1152
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// Byte offset of fp16 chunk j (8 elements) of row r in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int j) { return (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4); }


template <int EPI, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, const TcParams p) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ppdev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * C::STAGE_BYTES;
  auto full_b = [&](int s) { return bars + 8 * s; };
  auto ready_b = [&](int s) { return bars + 8 * (STAGES + s); };
  auto empty_b = [&](int s) { return bars + 8 * (2 * STAGES + s); };
  auto accf_b = [&](int b) { return bars + 8 * (3 * STAGES + b); };
  auto acce_b = [&](int b) { return bars + 8 * (3 * STAGES + 2 + b); };
  const uint32_t done_b = bars + 8 * (3 * STAGES + 4);
  const uint32_t tmem_slot = bars + 8 * (3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 8 - base));
  float* const ws_s = reinterpret_cast<float*>(gbase + STAGES * C::STAGE_BYTES + 256);  // [2][BN] weight scales
  float* const epi_s = ws_s + 2 * BN;  // [drain warps][32 rows][EPI_LD] epilogue staging
  auto sA = [&](int s) { return base + s * C::STAGE_BYTES; };
  auto sB = [&](int s) { return base + s * C::STAGE_BYTES + A_BYTES; };
  auto sW = [&](int s) { return base + s * C::STAGE_BYTES + A_BYTES + C::B_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int nkb = p.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(ready_b(s), 2 * N_CONV_WARPS);
      mbar_init(empty_b(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_b(b), 1);
      mbar_init(acce_b(b), 2 * N_DRAIN_WARPS);
    }
    mbar_init(done_b, 1);
    *abort_flag = 0;
    abort_flag[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));
  // The prologue above overlaps the previous kernel's tail; its results are read
  // from here on. With early_w the producer first issues the weight loads of the
  // stages it can fill without waiting (the model's weights, which no kernel of
  // the stream writes; a streamed layer's ring slot is waited for by a plain
  // stream-ordered launch before the layer's first kernel) and only then waits.
  ppdev::pdl_trigger();
  if (warp != 0) ppdev::pdl_wait();

  auto fail = [&]() {
    *abort_flag = 1;
    if (p.status) atomicExch(p.status, DEV_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_ROLE));
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int issued[STAGES] = {0};
      const Sched sc(p, cluster, n_clusters);
      // weights of the first STAGES k-blocks (every stage starts empty), then the wait
      int pre = 0;
      for (int u = 0; p.early_w && u < sc.units() && pre < STAGES; ++u) {
        int t, kb0, kb1;
        sc.unit(u, t, kb0, kb1);
        const int n_row = (t / p.num_m_tiles) * BN + (int)rank * (BN / 2);
        for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
          mbar_expect_tx(full_b(pre), A_BYTES + C::W_BYTES);
          tma_load_2d(sW(pre), &tmW, kb * BK, n_row, full_b(pre));
          issued[pre] = 1;
        }
      }
      ppdev::pdl_wait();
      int g = 0;  // k-blocks issued so far (the first `pre` have their weights in flight)
      for (int u = 0; u < sc.units() && !*abort_flag; ++u) {
        int t, kb0, kb1;
        sc.unit(u, t, kb0, kb1);
        const int m_row = (t % p.num_m_tiles) * 2 * BM + (int)rank * BM;
        const int n_row = (t / p.num_m_tiles) * BN + (int)rank * (BN / 2);
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          if (g < pre) {
            tma_load_2d(sA(s), &tmA, kb * BK, m_row, full_b(s));
          } else {
            if (!mbar_wait(empty_b(s), ph ^ 1, p.wait_cycles)) { fail(); break; }
            mbar_expect_tx(full_b(s), A_BYTES + C::W_BYTES);
            tma_load_2d(sA(s), &tmA, kb * BK, m_row, full_b(s));
            tma_load_2d(sW(s), &tmW, kb * BK, n_row, full_b(s));
            issued[s] = 1;
          }
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
      if (*abort_flag) {
        // let copies in flight land before the CTA's shared memory goes away
        for (int i = 0; i < STAGES; ++i) {
          const int st = (s + i) % STAGES;
          const uint32_t sph = (s + i >= STAGES) ? ph ^ 1 : ph;
          if (issued[st]) mbar_wait(full_b(st), sph ^ 1, p.wait_cycles);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_ROLE));
    if (rank == 0 && lane == 0 && !p.hold_mma) {
      const uint32_t idesc = idesc_f16(2 * BM, BN);
      int s = 0;
      uint32_t ph = 0;
      int g = 0;
      bool ok = true;
      const Sched sc(p, cluster, n_clusters);
      for (int u = 0; u < sc.units() && ok; ++u) {
        int t, ukb0, ukb1;
        sc.unit(u, t, ukb0, ukb1);
        for (int seg_k0 = ukb0; seg_k0 < ukb1 && ok; seg_k0 += p.seg_kb, ++g) {
          const int buf = g & 1;
          if (!mbar_wait(acce_b(buf), ((g >> 1) & 1) ^ 1, p.wait_cycles)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + buf * BN;
          const int kb0 = seg_k0, kb1 = min(ukb1, seg_k0 + p.seg_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(ready_b(s), ph, p.wait_cycles)) { fail(); ok = false; break; }
            tc_fence_after();
            const uint64_t da = umma_desc(sA(s)), db = umma_desc(sB(s));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA: advance 32 bytes inside the swizzle atom
              mma_f16_pair(d, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            mma_commit_pair(empty_b(s));
            if (++s == STAGES) { s = 0; ph ^= 1; }
          }
          if (ok) mma_commit_pair(accf_b(buf));
        }
      }
      if (!ok) {
        // let issued MMAs finish before the accumulator memory is released
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(done_b)
                     : "memory");
        mbar_wait(done_b, 0, p.wait_cycles);
      }
    }
  } else if (warp < CONV_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_ROLE));
  } else if (warp < DRAIN_WARP0) {
    // ---------------------------------------------------------------- converters
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CONV));
    const int et = threadIdx.x - 32 * CONV_WARP0;  // 0..127
    const Sched sc(p, cluster, n_clusters);
    int total_kb = 0;
    for (int u = 0; u < sc.units(); ++u) {
      int t, a, b;
      sc.unit(u, t, a, b);
      total_kb += b - a;
    }
    int s = 0;
    uint32_t ph = 0;
    for (int kb = 0; kb < total_kb; ++kb) {
      if (*abort_flag || !mbar_wait(full_b(s), ph, p.wait_cycles)) { fail(); break; }
      // widen this CTA's BN/2 weight rows x 64 k of int8 to fp16, UMMA layout
      uint8_t* bt = gbase + (sB(s) - base);
      const uint8_t* wt = gbase + (sW(s) - base);
#pragma unroll
      for (int i = 0; i < BN / 64; ++i) {
        const int c = et + 128 * i;  // 16-byte int8 chunk: row c/4, k = 16*(c%4) ..
        const int r = c >> 2, q = c & 3;
        const uint4 w = *reinterpret_cast<const uint4*>(wt + r * 64 + q * 16);
        uint4 o0, o1;
        i8x4_to_f16x4(w.x, o0.x, o0.y);
        i8x4_to_f16x4(w.y, o0.z, o0.w);
        i8x4_to_f16x4(w.z, o1.x, o1.y);
        i8x4_to_f16x4(w.w, o1.z, o1.w);
        *reinterpret_cast<uint4*>(bt + sw128(r, 2 * q)) = o0;
        *reinterpret_cast<uint4*>(bt + sw128(r, 2 * q + 1)) = o1;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(ready_b(s), 0);
      if (++s == STAGES) { s = 0; ph ^= 1; }
    }
  } else {
    // ---------------------------------------------------------------- drains + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_DRAIN));
    constexpr int COLS = C::COLS;
    const int et = threadIdx.x - 32 * DRAIN_WARP0;  // 0..255
    const int quarter = warp & 3;                   // TMEM lanes 32*quarter .. +31
    const int colq = (warp - DRAIN_WARP0) >> 2;     // accumulator columns COLS*colq .. +COLS-1
    int32_t run[COLS];
    volatile int* last_flag = abort_flag + 1;

    // Fold segment g's complete f32 accumulator into the int32 running sums.
    auto drain = [&](int g, bool first) {  // `first`: the unit's first segment starts the running sums
      const int buf = g & 1;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * BN + colq * COLS;
#pragma unroll
      for (int c = 0; c < COLS / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(taddr + c * 16, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int v = __float2int_rn(__uint_as_float(r[i]));
          run[c * 16 + i] = first ? v : run[c * 16 + i] + v;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_b(buf), 0);
    };

    // After the CTA's last unit is drained its pipeline stages are idle. There
    // the other contributors' partial sums and the epilogue's residual rows are
    // brought in with cp.async, every copy of a batch in flight at once, instead
    // of register loads that wait on L2 chunk by chunk. Each drain warp owns one
    // region, used by its partial slots and then by its residual rows.
    constexpr int XLD = COLS + 4;  // padded row of a warp's staged residual rows
    constexpr int PARK_BYTES = (COLS * 128 > 32 * XLD * 4) ? COLS * 128 : 32 * XLD * 4;
    static_assert(N_DRAIN_WARPS * PARK_BYTES <= STAGES * C::STAGE_BYTES, "parking fits in the stages");
    uint8_t* const park = gbase + (size_t)(warp - DRAIN_WARP0) * PARK_BYTES;
    int4* const park_i4 = reinterpret_cast<int4*>(park);  // [COLS/4][32 lanes]
    float* const park_x = reinterpret_cast<float*>(park);  // [32 rows][XLD]

    // Stream-K: this CTA's partial sums of `tile` meet the other contributors'.
    // Returns true for the last contributor, whose run[] then holds the totals.
    // parked: this is the CTA's last unit (the stages are free).
    auto finish_partial = [&](int tile, bool parked) -> bool {
      const int c_first = (int)(((long long)tile * nkb) / p.ipc);
      const int c_last = (int)((((long long)tile + 1) * nkb - 1) / p.ipc);
      const int n_contrib = c_last - c_first + 1;
      // slot layout [tile][slot][cta][drain warp][COLS/4][32 lanes] of int4: the j-th
      // store (or load) of a warp covers 512 contiguous bytes
      const int dw = warp - DRAIN_WARP0;
      auto slot_ptr = [&](int slot) {
        return reinterpret_cast<int4*>(p.part) +
               ((((size_t)tile * p.max_slots + slot) * 2 + rank) * N_DRAIN_WARPS + dw) * (COLS / 4) * 32 + lane;
      };
      // When every other contributor has already arrived (the usual case for the
      // tile's first k-blocks, which a cluster runs last), this CTA is the last
      // one and its own sums never leave its registers.
      if (et == 0) {
        int arrived;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(arrived) : "l"(p.cnt + 2 * tile + rank) : "memory");
        *last_flag = arrived == n_contrib - 1;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * N_DRAIN_WARPS) : "memory");
      if (!*last_flag) {  // (the flag is rewritten only after the next barrier, which every thread reaches after reading it)
        int4* mine = slot_ptr(cluster - c_first);
#pragma unroll
        for (int j = 0; j < COLS / 4; ++j)
          mine[32 * j] = make_int4(run[4 * j], run[4 * j + 1], run[4 * j + 2], run[4 * j + 3]);
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(32 * N_DRAIN_WARPS) : "memory");
        if (et == 0) *last_flag = atomicAdd(p.cnt + 2 * tile + rank, 1) == n_contrib - 1;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * N_DRAIN_WARPS) : "memory");
        if (!*last_flag) return false;
      }
      __threadfence();
      for (int sl = 0; sl < n_contrib; ++sl) {
        if (sl == cluster - c_first) continue;
        const int4* other = slot_ptr(sl);
        if (parked) {
          // each lane copies and then reads back only its own 16-byte pieces
#pragma unroll 8
          for (int j = 0; j < COLS / 4; ++j) ppdev::cp_async16(park_i4 + 32 * j + lane, other + 32 * j, 16);
          ppdev::cp_async_commit();
          ppdev::cp_async_wait<0>();
        }
#pragma unroll
        for (int j = 0; j < COLS / 4; ++j) {
          const int4 v = parked ? park_i4[32 * j + lane] : __ldcg(other + 32 * j);
          run[4 * j] += v.x;
          run[4 * j + 1] += v.y;
          run[4 * j + 2] += v.z;
          run[4 * j + 3] += v.w;
        }
      }
      if (et == 0) p.cnt[2 * tile + rank] = 0;  // ready for the next launch
      return true;
    };

    // Epilogue of a finished tile in chunks of 16 output columns (32 accumulator
    // columns for SwiGLU): (float(acc) * w_scale) * a_scale, then store,
    // residual add or SwiGLU. Rows past M are skipped. wsv: this warp's COLS
    // weight scales in shared memory; a_s: the row's activation scale.
    // The warp's 32 rows x 16 output columns of a chunk go through its own
    // slice of shared memory and leave as 8 rows x 64 bytes per store
    // instruction (16 full 32-byte sectors), instead of one 16-byte piece of
    // each of 32 rows; residual rows are loaded in the same pattern.
    float* const stg = epi_s + (warp - DRAIN_WARP0) * (32 * EPI_LD);
    auto epilogue = [&](int row0, int n0, const float* wsv, float a_s, bool parked) {  // row0: the warp's first row
      const int row = row0 + lane;
      if (EPI == EPI_ACC) {
        if (row >= p.M) return;
#pragma unroll
        for (int c = 0; c < COLS / 16; ++c) {
          int4* dst = reinterpret_cast<int4*>(p.acc_out + (size_t)row * p.N + n0 + 16 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_int4(run[16 * c + 4 * k], run[16 * c + 4 * k + 1], run[16 * c + 4 * k + 2], run[16 * c + 4 * k + 3]);
        }
        return;
      }
      if (EPI == EPI_ROPE) {
        // RoPE + K/V write. A 16-column chunk starts at a multiple of 16, so it lies
        // in one head; in a q or k head its columns are the pairs (j, j + hd/2) for
        // 8 consecutive j. The warp's 32 rows x 16 columns go through its staging
        // slice; lane (rq, cq) then rotates 2 pairs of row 8 it + rq and stores them
        // as 8 bytes at dims j and j + hd/2 (8 rows x 32 bytes per instruction).
        const TcRope& rp = p.rope;
        const int hd = rp.hd, half = hd >> 1, nqk = (rp.H + rp.Hkv) * hd;
        const int rq = lane >> 2, cq = lane & 3;
        // (cos, sin) of the lane's 2 pairs in each of its 4 rows, read one chunk
        // ahead through the read-only path (rows past M read the last row's entries)
        auto load_tab = [&](int c, float4 (&t)[4]) {
          const int col = n0 + 16 * c;
          if (col >= nqk) return;
          const int j = ((col % hd) >> 1) + 2 * cq;
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int pos = rp.pos0 + min(row0 + 8 * it + rq, p.M - 1);
            t[it] = __ldg(reinterpret_cast<const float4*>(rp.table + ((size_t)pos * half + j) * 2));
          }
        };
        float4 tnext[4];
        load_tab(0, tnext);
#pragma unroll
        for (int c = 0; c < COLS / 16; ++c) {
          float4 tc[4];
#pragma unroll
          for (int it = 0; it < 4; ++it) tc[it] = tnext[it];
          if (c + 1 < COLS / 16) load_tab(c + 1, tnext);
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = ppdev::dequant(run[16 * c + i], wsv[16 * c + i], a_s);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4*>(stg + lane * EPI_LD + 4 * k) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
          __syncwarp();
          const int col = n0 + 16 * c;
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int r = 8 * it + rq, row_r = row0 + r;
            const float4 x = *reinterpret_cast<const float4*>(stg + r * EPI_LD + 4 * cq);
            if (row_r >= p.M) continue;
            const int pos = rp.pos0 + row_r;
            if (col < nqk) {
              const int head = col / hd, j = ((col % hd) >> 1) + 2 * cq;
              const float4 t = tc[it];
              const float2 r0 = ppdev::rope_rot(x.x, x.y, make_float2(t.x, t.y));
              const float2 r1 = ppdev::rope_rot(x.z, x.w, make_float2(t.z, t.w));
              float* dst = head < rp.H ? rp.q_out + ((size_t)row_r * rp.H + head) * hd
                                       : rp.k_cache + ((size_t)pos * rp.Hkv + (head - rp.H)) * hd;
              *reinterpret_cast<float2*>(dst + j) = make_float2(r0.x, r1.x);
              *reinterpret_cast<float2*>(dst + j + half) = make_float2(r0.y, r1.y);
            } else {
              *reinterpret_cast<float4*>(rp.v_cache + (size_t)pos * rp.Hkv * hd + (col - nqk) + 4 * cq) = x;
            }
          }
          __syncwarp();  // the slice is free for the next chunk
        }
        return;
      }
      constexpr int CHUNKS = EPI == EPI_SWIGLU ? COLS / 32 : COLS / 16;
      const int ocol0 = EPI == EPI_SWIGLU ? n0 / 2 : n0;  // first output column of the warp
      // (only for wide tiles: with 4 chunks or fewer the one-chunk-ahead loads measured as fast)
      parked = parked && COLS >= 128;
      if (EPI == EPI_RESID && parked) {
        // the warp's 32 rows x COLS residual columns in one batch (rows past M are zero-filled)
        __syncwarp();  // every lane is done with the partial slots in this region
        for (int e = lane; e < 32 * (COLS / 4); e += 32) {
          const int r = e / (COLS / 4), c4 = e % (COLS / 4);
          const bool in = row0 + r < p.M;
          ppdev::cp_async16(park_x + r * XLD + 4 * c4, p.out + (size_t)(in ? row0 + r : row0) * p.ldo + ocol0 + 4 * c4,
                            in ? 16 : 0);
        }
        ppdev::cp_async_commit();
        ppdev::cp_async_wait<0>();
        __syncwarp();  // lanes read rows that other lanes copied
      }
#pragma unroll
      for (int c = 0; c < CHUNKS; ++c) {
        float v[16];
        if (EPI == EPI_SWIGLU) {
          // accumulator columns come in blocks of 16 gate rows then 16 up rows
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int cg = 32 * c + i;
            v[i] = ppdev::silu_mul(ppdev::dequant(run[cg], wsv[cg], a_s), ppdev::dequant(run[cg + 16], wsv[cg + 16], a_s));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = ppdev::dequant(run[16 * c + i], wsv[16 * c + i], a_s);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<float4*>(stg + lane * EPI_LD + 4 * k) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        __syncwarp();
        // lane -> row it*8 + lane/4, 16 bytes at column 4*(lane%4) of the chunk
        const int rq = lane >> 2, cq = lane & 3;
        float4 o[4], x[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int r = 8 * it + rq;
          o[it] = *reinterpret_cast<const float4*>(stg + r * EPI_LD + 4 * cq);
          if (EPI == EPI_RESID && row0 + r < p.M)
            x[it] = parked ? *reinterpret_cast<const float4*>(park_x + r * XLD + 16 * c + 4 * cq)
                           : *reinterpret_cast<const float4*>(p.out + (size_t)(row0 + r) * p.ldo + ocol0 + 16 * c + 4 * cq);
        }
        __syncwarp();  // the slice is free for the next chunk
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int r = 8 * it + rq;
          if (row0 + r >= p.M) continue;
          float4 w = o[it];
          if (EPI == EPI_RESID)
            w = make_float4(__fadd_rn(x[it].x, w.x), __fadd_rn(x[it].y, w.y), __fadd_rn(x[it].z, w.z), __fadd_rn(x[it].w, w.w));
          *reinterpret_cast<float4*>(p.out + (size_t)(row0 + r) * p.ldo + ocol0 + 16 * c + 4 * cq) = w;
        }
      }
    };

    const Sched sc(p, cluster, n_clusters);
    int g = 0;  // segments drained so far (selects the accumulator buffer and its phase)
    bool ok = true;
    for (int u = 0; u < sc.units() && ok; ++u) {
      int t, kb0, kb1;
      sc.unit(u, t, kb0, kb1);
      const int row = (t % p.num_m_tiles) * 2 * BM + (int)rank * BM + quarter * 32 + lane;
      // scales for the epilogue, loaded now so their latency hides behind the mainloop
      const int ncol = (t / p.num_m_tiles) * BN + et;  // et < BN: this thread's weight scale of the tile
      const float ws_r = (EPI != EPI_ACC && et < BN && ncol < p.N) ? __ldg(p.ws + ncol) : 0.f;
      const float as_r = (EPI != EPI_ACC && row < p.M) ? __ldg(p.as + row) : 0.f;
      for (int k0 = kb0; k0 < kb1; k0 += p.seg_kb, ++g) {
        if (*abort_flag || !mbar_wait(accf_b(g & 1), (g >> 1) & 1, p.wait_cycles)) { fail(); ok = false; break; }
        drain(g, k0 == kb0);
      }
      if (!ok) break;
      float* wsb = ws_s + (u & 1) * BN;  // two buffers: unit u+1 writes the other one
      if (et < BN) wsb[et] = ws_r;
      asm volatile("bar.sync 2, %0;" ::"n"(32 * N_DRAIN_WARPS) : "memory");
      const bool whole = kb0 == 0 && kb1 == nkb;
      const bool parked = u == sc.units() - 1;  // every MMA of the cluster is done: the stages are free
      if (whole || finish_partial(t, parked))
        epilogue(row - lane, (t / p.num_m_tiles) * BN + colq * COLS, wsb + colq * COLS, as_r, parked);
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Co-resident CTA pairs of the widest configuration (one pair per 2 SMs).
int max_clusters() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device(cache, [] {
    using C = Cfg<256>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.numAttrs = 0;  // the kernel declares its cluster shape
    int c = 0;
    cudaFuncSetAttribute(k_gemm_tc<EPI_STORE, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (cudaOccupancyMaxActiveClusters(&c, k_gemm_tc<EPI_STORE, 256>, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      c = sms / 2;
    }
    return c;
  });
}

template <int EPI, int BN>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mw, const TcParams& p, int clusters, cudaStream_t s,
                     bool pdl) {
  using C = Cfg<BN>;
  static std::atomic<uint64_t> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(k_gemm_tc<EPI, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl_if(pdl, k_gemm_tc<EPI, BN>, dim3(2 * clusters), dim3(THREADS), (size_t)C::SMEM_BYTES, s, ma, mw, p);
}

template <int EPI>
cudaError_t launch_bn(int bn, const CUtensorMap& ma, const CUtensorMap& mw, const TcParams& p, int clusters,
                      cudaStream_t s, bool pdl) {
  if (bn == 256) return launch_t<EPI, 256>(ma, mw, p, clusters, s, pdl);
  if (bn == 192) return launch_t<EPI, 192>(ma, mw, p, clusters, s, pdl);
  if (bn == 128) return launch_t<EPI, 128>(ma, mw, p, clusters, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace

bool tc_available() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3 && encoder() != nullptr;
}

cudaError_t make_tmap_a(CUtensorMap* map, const __half* a16, int rows, int k) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a16), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_w(CUtensorMap* map, const int8_t* w, int n, int k, int bn) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  if (bn != 256 && bn != 192 && bn != 128) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)k};
  cuuint32_t box[2] = {BK, (cuuint32_t)(bn / 2)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(w), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tile width for an m x n x k GEMM. A shape with too few tiles to fill the CTA
// pairs but enough k-blocks for stream-K (at least MIN_SK_KB per pair at width
// 256) runs stream-K at width 256. The mainloop is bound by shared-memory
// bandwidth (per k-block and CTA: TMA writes, the converter's int8 read and
// fp16 write, the tensor core's reads of the 16 KB activation tile and of both
// weight halves: 64 / 80 / 96 KB at widths 128 / 192 / 256, against 128 bytes
// per clock); the activation tile costs the same at every width, so a 256-row
// tile runs at the tensor core's rate while a 128-row tile reaches ~68% of it.
// Otherwise the width whose waves of tiles over the pairs cost the fewest
// weight columns per pair (ceil(tiles / pairs) x width); ties go to the wider
// tile. `wide` (other streams fill the pairs a launch leaves idle): the widest
// tile that divides n and no stream-K, the least SM time per GEMM.
int tc_bn(int m, int n, int k, bool wide) {
  const int mc = max_clusters();
  const int nmt = (m + 2 * BM - 1) / (2 * BM);
  if (wide) {
    for (int bn : {256, 192, 128})
      if (n % bn == 0) return bn;
    return 0;
  }
  if (n % 256 == 0) {
    const long long tiles = (long long)nmt * (n / 256), total = tiles * (k / BK);
    if (tiles < 2 * mc && total >= 2 * mc && (total + mc - 1) / mc >= MIN_SK_KB) return 256;
  }
  int best = 0;
  long long best_cost = 0;
  for (int bn : {256, 192, 128}) {
    if (n % bn) continue;
    const long long tiles = (long long)nmt * (n / bn);
    const long long cost = (tiles + mc - 1) / mc * bn;
    if (!best || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

namespace {

// Stream-K plan of one GEMM (ipc == 0: whole tiles round robin).
struct Plan {
  int bn, num_tiles, clusters, ipc, max_slots;
  size_t part_elems;
};

Plan plan(int m, int n, int k, bool wide) {
  Plan pl{};
  pl.bn = tc_bn(m, n, k, wide);
  if (!pl.bn) return pl;
  const int nmt = (m + 2 * BM - 1) / (2 * BM);
  const int nkb = k / BK;
  pl.num_tiles = nmt * (n / pl.bn);
  const int mc = max_clusters();
  if (wide || pl.num_tiles >= 2 * mc || pl.num_tiles * nkb < 2 * mc) {
    pl.clusters = std::min(pl.num_tiles, mc);
    return pl;
  }
  const long long total = (long long)pl.num_tiles * nkb;
  pl.ipc = std::max((int)((total + mc - 1) / mc), MAX_SEG_KB);  // at least one exact segment per cluster
  if (pl.ipc < MIN_SK_KB) {  // too little work per cluster to amortise a partial-tile fixup
    pl.ipc = 0;
    pl.clusters = std::min(pl.num_tiles, mc);
    return pl;
  }
  pl.clusters = (int)((total + pl.ipc - 1) / pl.ipc);
  pl.max_slots = (nkb + pl.ipc - 1) / pl.ipc + 1;
  pl.part_elems = (size_t)pl.num_tiles * pl.max_slots * 2 * BM * pl.bn;
  return pl;
}

}  // namespace

void tc_workspace_need(int m, int n, int k, size_t* part_bytes, size_t* counters) {
  const Plan pl = plan(m, n, k, false);
  *part_bytes = pl.part_elems * sizeof(int32_t);
  *counters = pl.ipc ? (size_t)pl.num_tiles * 2 : 0;
}

cudaError_t launch_gemm_tc(int epi, const CUtensorMap& ma, const CUtensorMap& mw, int bn, const float* ws,
                           const float* as, int m, int n, int k, float* out, int ldo, int32_t* acc, int seg_k,
                           int* status, const TcWorkspace& wsp, cudaStream_t s, const TcWaits& waits,
                           const TcRope& rope, bool wide, bool pdl, bool early_w) {
  TcParams p{};
  p.early_w = early_w ? 1 : 0;
  p.wait_cycles = waits.cycles;
  p.hold_mma = waits.hold_mma;
  p.M = m;
  p.N = n;
  p.K = k;
  p.seg_kb = std::max(1, std::min(MAX_SEG_KB, seg_k / BK));
  p.num_m_tiles = (m + 2 * BM - 1) / (2 * BM);
  p.ws = ws;
  p.as = as;
  p.out = out;
  p.ldo = ldo;
  p.acc_out = acc;
  p.status = status;
  p.rope = rope;
  Plan pl = plan(m, n, k, wide);
  if (!pl.bn || pl.bn != bn) return cudaErrorInvalidValue;  // the weight map was made for another tile width
  p.num_tiles = pl.num_tiles;
  if (pl.ipc && wsp.part && wsp.cnt && wsp.part_bytes >= pl.part_elems * sizeof(int32_t) &&
      wsp.counters >= (size_t)pl.num_tiles * 2) {
    p.ipc = pl.ipc;
    p.max_slots = pl.max_slots;
    p.part = wsp.part;
    p.cnt = wsp.cnt;
  } else {
    pl.clusters = std::min(pl.num_tiles, max_clusters());  // no workspace: whole tiles
  }
  switch (epi) {
    case EPI_STORE: return launch_bn<EPI_STORE>(bn, ma, mw, p, pl.clusters, s, pdl);
    case EPI_RESID: return launch_bn<EPI_RESID>(bn, ma, mw, p, pl.clusters, s, pdl);
    case EPI_SWIGLU: return launch_bn<EPI_SWIGLU>(bn, ma, mw, p, pl.clusters, s, pdl);
    case EPI_ACC: return launch_bn<EPI_ACC>(bn, ma, mw, p, pl.clusters, s, pdl);
    case EPI_ROPE:
      if (!rope.table || !rope.q_out || !rope.k_cache || !rope.v_cache || rope.hd % 16 ||
          n != (rope.H + 2 * rope.Hkv) * rope.hd)
        return cudaErrorInvalidValue;
      return launch_bn<EPI_ROPE>(bn, ma, mw, p, pl.clusters, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pp
