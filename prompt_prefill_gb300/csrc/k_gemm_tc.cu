// Exact int8 x int8 -> int32 GEMM on the 5th-generation tensor cores.
//
// "Batched Prefill", "The Solution": each weight row is dotted against the
// whole chunk of token columns, with activations quantised once per chunk.
// sm_103a has no integer tcgen05 MMA kind, so the integer GEMM runs on
// tcgen05.mma.kind::f16 with operands that hold the int8 codes exactly:
//   - every integer in [-127, 127] is an fp16 value, and so is every product
//     (|a*w| <= 16129 < 2^11 * 2^... fits the 22-bit product of two 11-bit
//     significands);
//   - an f32 sum of such products is exact while every partial sum stays below
//     2^24 in magnitude, i.e. for up to floor(2^24 / 127^2) = 1040 products.
// The K axis is therefore cut into segments of at most 1024 (16 k-blocks of
// 64); each segment accumulates into its own f32 TMEM buffer, which the
// epilogue warps read back, convert to int32 (exact) and add to int32
// registers. The result equals the int32 dot product bit for bit.
//
// Layout: a CTA pair (cluster of 2, cta_group::2) computes a 256-token x
// 256-weight-row tile; each CTA holds 128 token rows of A (fp16 codes, TMA,
// 128-byte swizzle) and 128 weight rows of B. Weights stay int8 in HBM: TMA
// brings int8 rows into shared memory and 8 converter warps widen them to
// fp16 in the UMMA K-major 128-byte-swizzled layout (exponent-bias method:
// 0x6400 | (b ^ 0x80) is the fp16 number 1024 + 128 + b, minus 1152 gives b).
// Warp 0 issues TMA, warp 1 (leader CTA) issues the MMAs, warps 4-11 convert
// and run the epilogue, each thread holding 128 int32 running sums (register
// split by setmaxnreg). Converter warps never block on the MMA: they drain a
// segment only once its accumulator is complete (polled between conversions)
// and emit a finished tile's epilogue in chunks between the next tile's
// conversions, so the stages ahead of the tensor core stay filled. Persistent over tiles; two TMEM accumulators of 256 columns alternate
// between segments. Every mbarrier wait is bounded: on
// expiry the kernel records a timeout in the status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int BM = 128;             // token rows per CTA (256 per pair)
constexpr int BN = 256;             // weight rows per pair tile (128 per CTA)
constexpr int BK = 64;              // k per stage: 128 bytes of fp16
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = (BN / 2) * BK * 2;    // 16 KB, converted weights
constexpr int W_BYTES = (BN / 2) * BK;        // 8 KB, int8 weights
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + W_BYTES;
constexpr int N_CONV_WARPS = 8;         // 2 per TMEM lane quarter, 128 accumulator columns each
constexpr int THREADS = 384;            // warpgroup 0: TMA, MMA, 2 idle; warpgroups 1-2: converters
constexpr int CONV_WARP0 = 4;
// Register split (setmaxnreg): launched at 168 per thread (12 x 32 x 168 = 64512 in the
// pool); warpgroup 0 drops to 40 and the converter warpgroups rise to 232:
// 4 x 32 x 40 + 8 x 32 x 232 = 64512, and per SM sub-partition (40 + 232 + 232) x 32 <= 16384.
constexpr int REGS_ROLE = 40, REGS_CONV = 232;
constexpr int TMEM_COLS = 512;
constexpr int MAX_SEG_KB = 16;      // 16 x 64 = 1024 products per exact f32 segment
constexpr int MIN_SK_KB = 64;       // stream-K only when each cluster owns >= 64 k-blocks (measured: fixups
                                    // cost more than they recover at ~40 k-blocks per cluster)
constexpr int EPI_EVERY = 2;        // conversions between two epilogue chunks of a finished tile
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz

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
  // space; partial tiles meet in `part` (int32 [tile][slot][cta][128][256]) and the
  // last contributor, counted in `cnt` ([tile][cta], zero between launches), adds
  // the partial sums and runs the epilogue. ipc == 0: whole tiles round robin.
  int ipc;
  int max_slots;
  int32_t* part;
  int* cnt;
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
// Non-blocking test of a barrier phase (lane 0 tests, the warp agrees).
__device__ __forceinline__ bool mbar_test_warp(uint32_t a, uint32_t parity) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Bounded wait: false after ~2 s without the phase completing.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
  if (mbar_try(a, parity)) return true;
  const long long end = clock64() + WAIT_CYCLES;
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

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ppdev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * STAGE_BYTES;
  auto full_b = [&](int s) { return bars + 8 * s; };
  auto ready_b = [&](int s) { return bars + 8 * (STAGES + s); };
  auto empty_b = [&](int s) { return bars + 8 * (2 * STAGES + s); };
  auto accf_b = [&](int b) { return bars + 8 * (3 * STAGES + b); };
  auto acce_b = [&](int b) { return bars + 8 * (3 * STAGES + 2 + b); };
  const uint32_t done_b = bars + 8 * (3 * STAGES + 4);
  const uint32_t tmem_slot = bars + 8 * (3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 8 - base));
  auto sA = [&](int s) { return base + s * STAGE_BYTES; };
  auto sB = [&](int s) { return base + s * STAGE_BYTES + A_BYTES; };
  auto sW = [&](int s) { return base + s * STAGE_BYTES + A_BYTES + B_BYTES; };

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
      mbar_init(acce_b(b), 2 * N_CONV_WARPS);
    }
    mbar_init(done_b, 1);
    *abort_flag = 0;
    abort_flag[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));

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
      for (int u = 0; u < sc.units() && !*abort_flag; ++u) {
        int t, kb0, kb1;
        sc.unit(u, t, kb0, kb1);
        const int m_row = (t % p.num_m_tiles) * 2 * BM + (int)rank * BM;
        const int n_row = (t / p.num_m_tiles) * BN + (int)rank * (BN / 2);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty_b(s), ph ^ 1)) { fail(); break; }
          mbar_expect_tx(full_b(s), A_BYTES + W_BYTES);
          tma_load_2d(sA(s), &tmA, kb * BK, m_row, full_b(s));
          tma_load_2d(sW(s), &tmW, kb * BK, n_row, full_b(s));
          issued[s] = 1;
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
      if (*abort_flag) {
        // let copies in flight land before the CTA's shared memory goes away
        for (int i = 0; i < STAGES; ++i) {
          const int st = (s + i) % STAGES;
          const uint32_t sph = (s + i >= STAGES) ? ph ^ 1 : ph;
          if (issued[st]) mbar_wait(full_b(st), sph ^ 1);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_ROLE));
    if (rank == 0 && lane == 0) {
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
          if (!mbar_wait(acce_b(buf), ((g >> 1) & 1) ^ 1)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + buf * 256;
          const int kb0 = seg_k0, kb1 = min(ukb1, seg_k0 + p.seg_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(ready_b(s), ph)) { fail(); ok = false; break; }
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
        mbar_wait(done_b, 0);
      }
    }
  } else if (warp < CONV_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_ROLE));
  } else {
    // ---------------------------------------------------------------- converters + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_CONV));
    const int et = threadIdx.x - 32 * CONV_WARP0;  // 0..255
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int colq = (warp - CONV_WARP0) >> 2;     // accumulator columns 128*colq .. +127
    int32_t run[128];
    int s = 0;
    uint32_t ph = 0;
    int done_kb = 0;      // k-blocks converted so far (all units)
    int next_seg = 0;     // segments drained so far (all units; selects the accumulator buffer)
    const Sched sc(p, cluster, n_clusters);
    const int n_units = sc.units();
    int total_kb = 0;
    for (int u = 0; u < n_units; ++u) {
      int t, a, b;
      sc.unit(u, t, a, b);
      total_kb += b - a;
    }
    // drain cursor: segment dseg of unit du, whose k-blocks start at conversion index dbase
    int du = 0, dseg = 0, dbase = 0, dtile = 0, dkb0 = 0, dkb1 = 0;
    if (n_units > 0) sc.unit(0, dtile, dkb0, dkb1);
    volatile int* last_flag = abort_flag + 1;

    // Fold segment g's complete f32 accumulator into the int32 running sums.
    auto drain = [&](int g, bool first) {  // `first`: the unit's first segment starts the running sums
      const int buf = g & 1;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * 256 + colq * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
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

    // Stream-K: this CTA's partial sums of `tile` meet the other contributors'.
    // Returns true for the last contributor, whose run[] then holds the totals.
    auto finish_partial = [&](int tile) -> bool {
      const int c_first = (int)(((long long)tile * nkb) / p.ipc);
      const int c_last = (int)((((long long)tile + 1) * nkb - 1) / p.ipc);
      const int n_contrib = c_last - c_first + 1;
      const int row = quarter * 32 + lane;
      auto slot_ptr = [&](int slot) {
        return p.part + ((((size_t)tile * p.max_slots + slot) * 2 + rank) * BM + row) * BN + colq * 128;
      };
      int4* mine = reinterpret_cast<int4*>(slot_ptr(cluster - c_first));
#pragma unroll
      for (int j = 0; j < 32; ++j) mine[j] = make_int4(run[4 * j], run[4 * j + 1], run[4 * j + 2], run[4 * j + 3]);
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(32 * N_CONV_WARPS) : "memory");
      if (et == 0) *last_flag = atomicAdd(p.cnt + 2 * tile + rank, 1) == n_contrib - 1;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * N_CONV_WARPS) : "memory");
      if (!*last_flag) return false;
      __threadfence();
      for (int sl = 0; sl < n_contrib; ++sl) {
        if (sl == cluster - c_first) continue;
        const int4* other = reinterpret_cast<const int4*>(slot_ptr(sl));
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int4 v = __ldcg(other + j);
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
    // residual add or SwiGLU. Rows past M are skipped.
    int epi_left = 0, epi_row0 = 0, epi_n0 = 0;
    constexpr int EPI_CHUNKS = EPI == EPI_SWIGLU ? 4 : 8;
    auto epi_chunk = [&](int c) {
      const int row = epi_row0 + lane;
      if (row >= p.M) return;
      if (EPI == EPI_ACC) {
        int4* dst = reinterpret_cast<int4*>(p.acc_out + (size_t)row * p.N + epi_n0 + 16 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_int4(run[16 * c + 4 * k], run[16 * c + 4 * k + 1], run[16 * c + 4 * k + 2], run[16 * c + 4 * k + 3]);
        return;
      }
      const float a_s = p.as[row];
      float v[16];
      if (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int cg = 32 * c + i;
          v[i] = ppdev::silu_mul(ppdev::dequant(run[cg], __ldg(p.ws + epi_n0 + cg), a_s),
                                 ppdev::dequant(run[cg + 16], __ldg(p.ws + epi_n0 + cg + 16), a_s));
        }
        float4* dst = reinterpret_cast<float4*>(p.out + (size_t)row * p.ldo + epi_n0 / 2 + 16 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = ppdev::dequant(run[16 * c + i], __ldg(p.ws + epi_n0 + 16 * c + i), a_s);
        float4* dst = reinterpret_cast<float4*>(p.out + (size_t)row * p.ldo + epi_n0 + 16 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
          if (EPI == EPI_RESID) {
            const float4 x = dst[k];
            o = make_float4(__fadd_rn(x.x, o.x), __fadd_rn(x.y, o.y), __fadd_rn(x.z, o.z), __fadd_rn(x.w, o.w));
          }
          dst[k] = o;
        }
      }
    };
    auto epi_next = [&]() {  // the next pending chunk (each branch has compile-time indices)
      const int c = EPI_CHUNKS - epi_left;
#pragma unroll
      for (int k = 0; k < EPI_CHUNKS; ++k)
        if (k == c) epi_chunk(k);
      --epi_left;
    };

    int since_epi = 0;
    long long idle_since = clock64();
    while (true) {
      bool progressed = false;
      const bool seg_done = du < n_units && dbase + min(dkb1 - dkb0, (dseg + 1) * p.seg_kb) - 1 < done_kb &&
                            mbar_test_warp(accf_b(next_seg & 1), (next_seg >> 1) & 1);
      if (seg_done && epi_left == 0) {
        drain(next_seg++, dseg == 0);
        ++dseg;
        if (dkb0 + dseg * p.seg_kb >= dkb1) {  // the unit is complete
          const bool whole = dkb0 == 0 && dkb1 == nkb;
          if (whole || finish_partial(dtile)) {  // queue the tile's epilogue
            epi_row0 = (dtile % p.num_m_tiles) * 2 * BM + (int)rank * BM + quarter * 32;
            epi_n0 = (dtile / p.num_m_tiles) * BN + colq * 128;
            epi_left = EPI_CHUNKS;
            since_epi = EPI_EVERY;
          }
          dbase += dkb1 - dkb0;
          dseg = 0;
          if (++du < n_units) sc.unit(du, dtile, dkb0, dkb1);
        }
        progressed = true;
      } else if (epi_left > 0 && (seg_done || since_epi >= EPI_EVERY || done_kb == total_kb)) {
        epi_next();  // a finished tile's sums must be written before the next drain reuses them
        since_epi = 0;
        progressed = true;
      } else if (done_kb < total_kb && mbar_test_warp(full_b(s), ph)) {
        // widen this CTA's 128 weight rows x 64 k of int8 to fp16, UMMA layout
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = et + 256 * i;  // 16-byte int8 chunk: row c/4, k = 16*(c%4) ..
          const int r = c >> 2, q = c & 3;
          const uint4 w = *reinterpret_cast<const uint4*>(gbase + (sW(s) - base) + r * 64 + q * 16);
          uint4 o0, o1;
          i8x4_to_f16x4(w.x, o0.x, o0.y);
          i8x4_to_f16x4(w.y, o0.z, o0.w);
          i8x4_to_f16x4(w.z, o1.x, o1.y);
          i8x4_to_f16x4(w.w, o1.z, o1.w);
          uint8_t* bt = gbase + (sB(s) - base);
          *reinterpret_cast<uint4*>(bt + sw128(r, 2 * q)) = o0;
          *reinterpret_cast<uint4*>(bt + sw128(r, 2 * q + 1)) = o1;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(ready_b(s), 0);
        if (++s == STAGES) { s = 0; ph ^= 1; }
        ++done_kb;
        ++since_epi;
        progressed = true;
      }
      if (done_kb == total_kb && du == n_units && epi_left == 0) break;
      if (progressed) {
        idle_since = clock64();
      } else {
        if (*abort_flag || clock64() - idle_since > WAIT_CYCLES) { fail(); break; }
        __nanosleep(20);
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
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

int max_clusters() {
  static int n = 0;
  if (!n) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 0;  // the kernel declares its cluster shape
    int c = 0;
    cudaFuncSetAttribute(k_gemm_tc<EPI_STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (cudaOccupancyMaxActiveClusters(&c, k_gemm_tc<EPI_STORE>, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      c = sms / 2;
    }
    n = c;
  }
  return n;
}

template <int EPI>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mw, const TcParams& p, int clusters, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_gemm_tc<EPI><<<2 * clusters, THREADS, SMEM_BYTES, s>>>(ma, mw, p);
  return cudaGetLastError();
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

cudaError_t make_tmap_w(CUtensorMap* map, const int8_t* w, int n, int k) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)k};
  cuuint32_t box[2] = {BK, BN / 2};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(w), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// Stream-K plan of one GEMM (ipc == 0: whole tiles round robin).
struct Plan {
  int num_tiles, clusters, ipc, max_slots;
  size_t part_elems;
};

Plan plan(int m, int n, int k) {
  Plan pl{};
  const int nmt = (m + 2 * BM - 1) / (2 * BM);
  const int nkb = k / BK;
  pl.num_tiles = nmt * (n / BN);
  const int mc = max_clusters();
  if (pl.num_tiles >= 2 * mc || pl.num_tiles * nkb < 2 * mc) {
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
  pl.part_elems = (size_t)pl.num_tiles * pl.max_slots * 2 * BM * BN;
  return pl;
}

}  // namespace

void tc_workspace_need(int m, int n, int k, size_t* part_bytes, size_t* counters) {
  const Plan pl = plan(m, n, k);
  *part_bytes = pl.part_elems * sizeof(int32_t);
  *counters = pl.ipc ? (size_t)pl.num_tiles * 2 : 0;
}

cudaError_t launch_gemm_tc(int epi, const CUtensorMap& ma, const CUtensorMap& mw, const float* ws, const float* as,
                           int m, int n, int k, float* out, int ldo, int32_t* acc, int seg_k, int* status,
                           const TcWorkspace& wsp, cudaStream_t s) {
  TcParams p{};
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
  Plan pl = plan(m, n, k);
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
    case EPI_STORE: return launch_t<EPI_STORE>(ma, mw, p, pl.clusters, s);
    case EPI_RESID: return launch_t<EPI_RESID>(ma, mw, p, pl.clusters, s);
    case EPI_SWIGLU: return launch_t<EPI_SWIGLU>(ma, mw, p, pl.clusters, s);
    case EPI_ACC: return launch_t<EPI_ACC>(ma, mw, p, pl.clusters, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pp
