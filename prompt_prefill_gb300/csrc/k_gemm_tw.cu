// Exact int8 x int8 -> int32 GEMM on the 5th-generation tensor cores for
// short chunks (up to 128 token rows): the weights are the MMA's M side.
//
// "Batched Prefill", "The Solution": each weight row is dotted against the
// whole chunk of token columns, with activations quantised once per chunk.
// As in k_gemm_tc.cu, the integer GEMM runs on tcgen05.mma.kind::f16 with fp16
// operands that hold the int8 codes exactly, and K is cut into exact f32
// segments of at most 1024 products drained into int32.
//
// Operands. A CTA pair (cluster of 2, cta_group::2) owns 256 weight rows, 128
// per CTA in its 128 TMEM lanes: TMA brings each CTA's int8 weight rows (64 k
// = 64 bytes per row, 64-byte swizzle) into shared memory, and converter
// warps, one thread per row, widen them to fp16 (the exponent-bias trick: the
// bytes b ^ 0x80 placed under the exponent byte 0x64 are the fp16 numbers
// 1152 + b, so subtracting 1152 leaves b exactly; the same construction as the
// widely used "fast int8 to fp16" permute-and-subtract conversion) and store
// them with tcgen05.st straight into a TMEM slot of the stage, from which the
// MMA reads them. The tokens are the N side: NT fp16 code rows per pair (NT/2
// per CTA, TMA, 128-byte swizzle). NT is 32, 64 or 128, the smallest that holds
// the chunk, so a chunk of 32 rows runs 256 x 32 tiles instead of the 256-row
// token tiles of k_gemm_tc.cu, of which it would use an eighth.
//
// Roles (16 warps): warp 0 issues the weight TMA, warp 2 the token TMA (one
// thread's TMA loads complete one after another, ~37 bytes per clock each on
// a GB300, while loads from different warps proceed in parallel), warp 1
// (leader CTA) issues the MMAs, warpgroup 1 converts, warpgroups 2-3 drain the
// accumulators and run the epilogue (each thread holds one weight row: NT/2
// int32 running sums). Persistent over tiles (256 weight rows x NT tokens);
// two TMEM accumulators of NT columns alternate between segments. Every
// mbarrier wait is bounded: on expiry the kernel records a timeout in the
// status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pp_internal.cuh"

namespace pp {
namespace {

constexpr int WM = 128;            // weight rows per CTA (256 per pair): the M side, in TMEM lanes
constexpr int BK = 64;             // k per stage
constexpr int W_BYTES = WM * BK;   // int8 weights of one CTA per stage (8 KB, 64-byte swizzle)
constexpr int A_COLS = BK / 2;     // TMEM columns of one converted stage (two fp16 per column)
constexpr int N_CONV_WARPS = 4;    // warpgroup 1: int8 -> fp16 into TMEM, one thread per weight row
constexpr int N_DRAIN_WARPS = 8;   // warpgroups 2-3: 2 per TMEM lane quarter, NT/2 token columns each
constexpr int THREADS = 512;       // warpgroup 0: TMA, MMA, 2 idle
constexpr int CONV_WARP0 = 4;
constexpr int DRAIN_WARP0 = 8;
constexpr int MAX_SEG_KB = 16;     // 16 x 64 = 1024 products per exact f32 segment
constexpr int MIN_SK_KB = 32;      // NT = 128: stream-K gives each cluster >= 32 k-blocks
// A CTA of the full form (NT = 128) allocates all 512 TMEM columns, so two of them must
// never share an SM (a pair would wait on another pair's columns): each asks for more than
// half of the SM's shared memory.
constexpr int MIN_SMEM = 120 * 1024;
constexpr int SMEM_SM = 233472;     // shared memory of an SM, 1 KB of it reserved per resident CTA

constexpr int BAR_BYTES = 1024;     // mbarriers, the TMEM address slot and two flags

// Per-token-tile constants. The int8 weights stream through a ring of W_STAGES shared-memory
// stages that the converters free as soon as they have read them (not when the MMA is done
// with the k-block, as the tokens and the converted weights in their TMEM slots are); a
// deeper weight ring (12-16 stages, all the shared memory) measured no faster.
// NT = 128: 8 stages, all 512 TMEM columns, one CTA per SM,
// registers launched at 128 per thread and split (setmaxnreg) 48 / 72 / 192 between
// warpgroup 0, the converters and the drains (up to 128 running sums and 64 accumulator
// columns in flight): 128 x 48 + 128 x 72 + 256 x 192 = 64512 of 65536. NT <= 64 (the lean
// form): a launch is a latency chain (weights streamed once, few MMAs), so two CTAs share
// an SM: 4 stages, 256 TMEM columns (two accumulators of NT plus four weight slots), no
// shared-memory floor, registers launched at 64 and split 40 / 64 / 72 (128 x 40 + 128 x 64
// + 256 x 72 = 31744 of the 32768 launched, half the file).
template <int NT>
struct Cfg {
  static constexpr bool LEAN = NT <= 64;
  static constexpr int STAGES = LEAN ? 4 : 8;            // token stages and TMEM weight slots
  static constexpr int W_STAGES = STAGES;                // int8 weight stages
  static constexpr int TMEM_COLS = LEAN ? 256 : 512;
  static constexpr int CTAS_PER_SM = LEAN ? 2 : 1;
  static constexpr int R_LAUNCH = 65536 / (THREADS * CTAS_PER_SM);  // registers per thread at launch
  static constexpr int R_ROLE = LEAN ? 40 : 48, R_CONV = LEAN ? 64 : 72, R_DRAIN = LEAN ? 72 : 192;
  static_assert(R_ROLE <= R_LAUNCH && R_CONV <= R_LAUNCH && R_DRAIN >= R_LAUNCH, "dec / dec / inc");
  static_assert(128 * R_ROLE + 128 * R_CONV + 256 * R_DRAIN <= R_LAUNCH * THREADS, "register split");
  static constexpr int TOK = NT / 2;                     // token rows per CTA
  static constexpr int T_BYTES = TOK * BK * 2;           // fp16 tokens of one CTA per stage
  static constexpr int W_RING = W_STAGES * W_BYTES, T_RING = STAGES * T_BYTES;
  static constexpr int COLS = NT / 2;                    // accumulator columns per drain warp
  static constexpr int TMEM_A0 = 2 * NT;                 // first column of the weight slots
  static_assert(TMEM_A0 + STAGES * A_COLS <= TMEM_COLS, "TMEM: two accumulators and the weight slots");
  static_assert(W_BYTES % 1024 == 0 && T_BYTES % 1024 == 0, "every stage keeps the 1024-byte swizzle atoms aligned");
  static constexpr int USED = W_RING + T_RING + 1024 /*align*/ + BAR_BYTES + 2 * NT * 4 /*token scales*/;
  static constexpr int SMEM_BYTES = (LEAN || USED > MIN_SMEM) ? USED : MIN_SMEM;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(CTAS_PER_SM * (SMEM_BYTES + 1024) <= SMEM_SM, "CTAs per SM by shared memory");
};

struct TcParams {
  int M, N, K;  // M tokens, N weight rows
  int seg_kb;
  int num_t_tiles, num_tiles;  // token tiles per weight tile; all tiles
  const float* ws;
  const float* as;
  float* out;
  int ldo;
  int32_t* acc_out;
  int* status;
  // stream-K: cluster c owns iterations [c*ipc, (c+1)*ipc) of the (tile, k-block)
  // space; partial tiles meet in `part` (int32 per slot and CTA) and the last
  // contributor, counted in `cnt` ([tile][cta], zero between launches), adds the
  // partial sums and runs the epilogue. ipc == 0: whole tiles round robin.
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
// the default (CTA-scope release) semantics. A cluster-scope release here costs
// a device-wide memory barrier per arrive; what the arrive hands over (tensor
// memory written and waited for with tcgen05.wait::st, or drained accumulator
// columns) is ordered by the tcgen05 fences around it.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t a, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
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
// Bounded wait: false after `limit` clock64 cycles without the phase completing.
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

// D[tmem] (+)= A[tmem] x B[smem]^T over the CTA pair (A: this CTA's 128 lanes, B: both CTAs' halves).
__device__ __forceinline__ void mma_f16_pair_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive once on barrier `a` in both CTAs of the pair when all prior MMAs of this thread complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t a) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(a),
      "h"((uint16_t)0x3)
      : "memory");
}

// 16 or 32 consecutive TMEM columns of this thread's lane -> r (no wait: one
// tcgen05.wait::ld covers every load issued before it, and each wait costs a
// TMEM round trip, so the drains issue a batch of loads per wait).
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane <- r[0..31].
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Four int8 codes -> two f16x2 words holding the same integers (lower k in the lower half).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;  // b + 128 as unsigned bytes
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));  // (1024 + 128 + b) - 1152
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

template <int EPI, int NT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, Cfg<NT>::CTAS_PER_SM)
    k_gemm_tw(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT, const TcParams p) {
  using C = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ppdev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bars = base + C::W_RING + C::T_RING;
  // full: one barrier per producer and stage (weight stage, token stage), so that a
  // producer that gives up can wait for exactly its own copies in flight; wfree: the
  // converters have read a weight stage; ready / empty: a token stage and its TMEM slot
  // are loaded and converted / read by the MMA.
  constexpr int WS = C::W_STAGES, TS = C::STAGES, NB0 = 2 * WS + 3 * TS;
  auto full_b = [&](int src, int s) { return bars + 8 * (src == 0 ? s : WS + s); };
  auto ready_b = [&](int s) { return bars + 8 * (WS + TS + s); };
  auto empty_b = [&](int s) { return bars + 8 * (WS + 2 * TS + s); };
  auto wfree_b = [&](int s) { return bars + 8 * (WS + 3 * TS + s); };
  auto accf_b = [&](int b) { return bars + 8 * (NB0 + b); };
  auto acce_b = [&](int b) { return bars + 8 * (NB0 + 2 + b); };
  const uint32_t done_b = bars + 8 * (NB0 + 4);
  const uint32_t tmem_slot = bars + 8 * (NB0 + 5);
  static_assert(8 * (NB0 + 6) + 8 <= BAR_BYTES, "barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 8 - base));
  float* const as_s = reinterpret_cast<float*>(gbase + C::W_RING + C::T_RING + BAR_BYTES);  // [2][NT] token scales
  auto sW = [&](int s) { return base + s * W_BYTES; };
  auto sT = [&](int s) { return base + C::W_RING + s * C::T_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int nkb = p.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < WS; ++s) {
      mbar_init(full_b(0, s), 1);
      mbar_init(wfree_b(s), N_CONV_WARPS);  // this CTA's converter warps
    }
    for (int s = 0; s < TS; ++s) {
      mbar_init(full_b(1, s), 1);
      mbar_init(ready_b(s), 2 * N_CONV_WARPS);
      mbar_init(empty_b(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_b(b), 1);
      mbar_init(acce_b(b), 2 * N_DRAIN_WARPS);  // every drain warp of both CTAs
    }
    mbar_init(done_b, 1);
    *abort_flag = 0;
    abort_flag[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(C::TMEM_COLS));
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

  if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------------- TMA producers
    // One thread per operand stream: warp 0 the weights, warp 2 the tokens.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::R_ROLE));
    if (lane == 0) {
      const int src = warp == 0 ? 0 : 1;  // 0 weights, 1 tokens
      const uint32_t bytes = src == 0 ? W_BYTES : C::T_BYTES;
      const int RS = src == 0 ? WS : TS;  // this stream's ring
      int s = 0;
      uint32_t ph = 0;
      int issued[WS > TS ? WS : TS] = {0};
      const Sched sc(p, cluster, n_clusters);
      int pre = 0;
      for (int u = 0; src == 0 && p.early_w && u < sc.units() && pre < WS; ++u) {
        int t, kb0, kb1;
        sc.unit(u, t, kb0, kb1);
        const int w_row = (t / p.num_t_tiles) * 2 * WM + (int)rank * WM;
        for (int kb = kb0; kb < kb1 && pre < WS; ++kb, ++pre) {
          mbar_expect_tx(full_b(0, pre), bytes);
          tma_load_2d(sW(pre), &tmW, kb * BK, w_row, full_b(0, pre));
          issued[pre] = 1;
        }
      }
      ppdev::pdl_wait();
      int g = 0;  // k-blocks issued so far (the first `pre` are already in flight)
      for (int u = 0; u < sc.units() && !*abort_flag; ++u) {
        int t, kb0, kb1;
        sc.unit(u, t, kb0, kb1);
        const int w_row = (t / p.num_t_tiles) * 2 * WM + (int)rank * WM;
        // CTA rank r holds token rows r * TOK .. + TOK of the tile
        const int t_row = (t % p.num_t_tiles) * NT + (int)rank * C::TOK;
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          if (g >= pre) {
            if (!mbar_wait(src == 0 ? wfree_b(s) : empty_b(s), ph ^ 1, p.wait_cycles)) { fail(); break; }
            mbar_expect_tx(full_b(src, s), bytes);
            if (src == 0)
              tma_load_2d(sW(s), &tmW, kb * BK, w_row, full_b(0, s));
            else
              tma_load_2d(sT(s), &tmT, kb * BK, t_row, full_b(1, s));
            issued[s] = 1;
          }
          if (++s == RS) { s = 0; ph ^= 1; }
        }
      }
      if (*abort_flag) {
        // let this stream's copies in flight land before the CTA's shared memory goes away
        for (int i = 0; i < RS; ++i) {
          const int st = (s + i) % RS;
          const uint32_t sph = (s + i >= RS) ? ph ^ 1 : ph;
          if (issued[st]) mbar_wait(full_b(src, st), sph ^ 1, p.wait_cycles);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::R_ROLE));
    if (rank == 0 && lane == 0 && !p.hold_mma) {
      const uint32_t idesc = idesc_f16(2 * WM, NT);
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
          const uint32_t d = tmem + buf * NT;
          const int kb0 = seg_k0, kb1 = min(ukb1, seg_k0 + p.seg_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(ready_b(s), ph, p.wait_cycles)) { fail(); ok = false; break; }
            tc_fence_after();
            const uint32_t a = tmem + C::TMEM_A0 + s * A_COLS;
            const uint64_t db = umma_desc(sT(s));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA: 8 TMEM columns, 32 bytes of the swizzle atom
              mma_f16_pair_ta(d, a + 8 * k, db + (uint64_t)(2 * k), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            mma_commit_pair(empty_b(s));
            if (++s == C::STAGES) { s = 0; ph ^= 1; }
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::R_ROLE));  // warp 3: idle
  } else if (warp < DRAIN_WARP0) {
    // ---------------------------------------------------------------- converters
    if (C::R_CONV < C::R_LAUNCH) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::R_CONV));
    const int row = threadIdx.x - 32 * CONV_WARP0;  // this thread's weight row of the CTA, = its TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + C::TMEM_A0;
    const uint32_t swz = (uint32_t)((row >> 1) & 3);  // 64-byte swizzle of the TMA tile: chunk c at c ^ swz
    const Sched sc(p, cluster, n_clusters);
    int total_kb = 0;
    for (int u = 0; u < sc.units(); ++u) {
      int t, a, b;
      sc.unit(u, t, a, b);
      total_kb += b - a;
    }
    int s = 0, sw = 0;  // token stage / TMEM slot, weight stage
    uint32_t ph = 0, phw = 0;
    for (int kb = 0; kb < total_kb; ++kb) {
      // this k-block's weights, and its tokens (the MMA reads them once the converters
      // arrive; their load was issued after the MMA had freed TMEM slot s)
      bool landed = !*abort_flag && mbar_wait(full_b(0, sw), phw, p.wait_cycles);
      landed = landed && mbar_wait(full_b(1, s), ph, p.wait_cycles);
      if (!landed) { fail(); break; }
      const uint8_t* wr = gbase + (sW(sw) - base) + row * 64;
      uint32_t f[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // k = 16c .. 16c + 15
        const uint4 w = *reinterpret_cast<const uint4*>(wr + 16 * (c ^ swz));
        i8x4_to_f16x4(w.x, f[8 * c + 0], f[8 * c + 1]);
        i8x4_to_f16x4(w.y, f[8 * c + 2], f[8 * c + 3]);
        i8x4_to_f16x4(w.z, f[8 * c + 4], f[8 * c + 5]);
        i8x4_to_f16x4(w.w, f[8 * c + 6], f[8 * c + 7]);
      }
      // every lane has read its row of the weight stage; order those generic-proxy reads
      // before the TMA (async proxy) write that refills the stage once it is free (without
      // this fence, with the weight ring running 12-16 stages ahead, a refill was seen to
      // overtake the reads under concurrent launches)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_local(wfree_b(sw));
      if (++sw == WS) { sw = 0; phw ^= 1; }
      tmem_st32(lane_addr + s * A_COLS, f);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(ready_b(s), 0);
      if (++s == TS) { s = 0; ph ^= 1; }
    }
  } else {
    // ---------------------------------------------------------------- drains + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::R_DRAIN));
    constexpr int COLS = C::COLS;
    const int et = threadIdx.x - 32 * DRAIN_WARP0;  // 0..255
    const int quarter = warp & 3;                   // TMEM lanes (weight rows) 32*quarter .. +31
    const int colh = (warp - DRAIN_WARP0) >> 2;     // accumulator columns (tokens) COLS*colh .. +COLS-1
    const int dw = warp - DRAIN_WARP0;
    int32_t run[COLS];
    volatile int* last_flag = abort_flag + 1;

    // Fold segment g's complete f32 accumulator (buffer g & 1) into the int32 running sums.
    auto drain = [&](int g, bool first) {  // `first`: the unit's first segment starts the running sums
      const int buf = g & 1;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * NT + colh * COLS;
      // batches of up to 64 columns per wait
      constexpr int BATCH = COLS < 64 ? COLS : 64;
#pragma unroll
      for (int c0 = 0; c0 < COLS; c0 += BATCH) {
        uint32_t r[BATCH];
        if (BATCH == 16) {
          tmem_ld16_nw(taddr + c0, r);
        } else {
#pragma unroll
          for (int j = 0; j < BATCH; j += 32) tmem_ld32_nw(taddr + c0 + j, r + j);
        }
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
          const int v = __float2int_rn(__uint_as_float(r[i]));
          run[c0 + i] = first ? v : run[c0 + i] + v;
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
      // slot layout [tile][slot][cta][drain warp][COLS/4][32 lanes] of int4: the j-th
      // store (or load) of a warp covers 512 contiguous bytes
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
#pragma unroll
        for (int j = 0; j < COLS / 4; ++j) {
          const int4 v = __ldcg(other + 32 * j);
          run[4 * j] += v.x;
          run[4 * j + 1] += v.y;
          run[4 * j + 2] += v.z;
          run[4 * j + 3] += v.w;
        }
      }
      if (et == 0) p.cnt[2 * tile + rank] = 0;  // ready for the next launch
      return true;
    };

    // Epilogue of a finished tile: this thread's weight row R and the warp's COLS
    // tokens t0 + i (rows past N or tokens past M are skipped). For each token the
    // warp's 32 lanes write 32 consecutive output columns (128 contiguous bytes).
    // a_s: the tile's token scales in shared memory, from the warp's first token.
    auto epilogue = [&](int R, int t0, float ws_r, const float* a_s) {
      const bool row_ok = R < p.N;
      if (EPI == EPI_ACC) {
        if (!row_ok) return;
#pragma unroll
        for (int i = 0; i < COLS; ++i)
          if (t0 + i < p.M) p.acc_out[(size_t)(t0 + i) * p.N + R] = run[i];
        return;
      }
      if (EPI == EPI_STORE) {
        if (!row_ok) return;
#pragma unroll
        for (int i = 0; i < COLS; ++i)
          if (t0 + i < p.M) p.out[(size_t)(t0 + i) * p.ldo + R] = ppdev::dequant(run[i], ws_r, a_s[i]);
        return;
      }
      if (EPI == EPI_RESID) {
        if (!row_ok) return;
        // residual rows in batches of 16 loads in flight
        constexpr int RB = 16;
#pragma unroll
        for (int i0 = 0; i0 < COLS; i0 += RB) {
          float x[RB];
#pragma unroll
          for (int i = 0; i < RB; ++i)
            x[i] = (t0 + i0 + i < p.M) ? p.out[(size_t)(t0 + i0 + i) * p.ldo + R] : 0.f;
#pragma unroll
          for (int i = 0; i < RB; ++i)
            if (t0 + i0 + i < p.M)
              p.out[(size_t)(t0 + i0 + i) * p.ldo + R] =
                  __fadd_rn(x[i], ppdev::dequant(run[i0 + i], ws_r, a_s[i0 + i]));
        }
        return;
      }
      if (EPI == EPI_SWIGLU) {
        // rows come in blocks of 16 gate rows then 16 up rows: lanes 0-15 hold the
        // gate rows of the warp's block, lanes 16-31 the matching up rows
        const int f = 16 * (R >> 5) + (lane & 15);
#pragma unroll
        for (int i = 0; i < COLS; ++i) {
          const float v = ppdev::dequant(run[i], ws_r, a_s[i]);
          const float u = __shfl_down_sync(0xffffffffu, v, 16);
          if (lane < 16 && row_ok && t0 + i < p.M) p.out[(size_t)(t0 + i) * p.ldo + f] = ppdev::silu_mul(v, u);
        }
        return;
      }
      if (EPI == EPI_ROPE) {
        // RoPE + K/V write. Rows of a q or k head are in pair order: row 2j + e of the
        // head is its dim j + e * hd/2, so a rotated pair sits in lanes (2j, 2j + 1).
        // Both lanes rotate the pair (x_j, x_{j+hd/2}) and keep their own half. A warp's
        // 32 rows lie in one head (hd is a multiple of 32).
        const TcRope& rp = p.rope;
        const int hd = rp.hd, half = hd >> 1, nqk = (rp.H + rp.Hkv) * hd;
        const int head = R / hd, rr = R % hd, j = rr >> 1, e = rr & 1;
        const bool qk = R < nqk;
#pragma unroll
        for (int i = 0; i < COLS; ++i) {
          const int t = t0 + i;
          const float v = ppdev::dequant(run[i], ws_r, a_s[i]);
          const float w = __shfl_xor_sync(0xffffffffu, v, 1);
          if (!row_ok || t >= p.M) continue;
          const int pos = rp.pos0 + t;
          if (qk) {
            const float2 cs = __ldg(reinterpret_cast<const float2*>(rp.table) + (size_t)pos * half + j);
            const float2 r2 = e ? ppdev::rope_rot(w, v, cs) : ppdev::rope_rot(v, w, cs);
            float* dst = head < rp.H ? rp.q_out + ((size_t)t * rp.H + head) * hd
                                     : rp.k_cache + ((size_t)pos * rp.Hkv + (head - rp.H)) * hd;
            dst[j + e * half] = e ? r2.y : r2.x;
          } else {
            rp.v_cache[(size_t)pos * rp.Hkv * hd + (R - nqk)] = v;
          }
        }
        return;
      }
    };

    const Sched sc(p, cluster, n_clusters);
    int g = 0;  // segments drained so far (selects the accumulator buffer and its phase)
    bool ok = true;
    for (int u = 0; u < sc.units() && ok; ++u) {
      int t, kb0, kb1;
      sc.unit(u, t, kb0, kb1);
      const int R = (t / p.num_t_tiles) * 2 * WM + (int)rank * WM + quarter * 32 + lane;  // this thread's weight row
      const int tok0 = (t % p.num_t_tiles) * NT;                                            // the tile's first token
      // scales for the epilogue, loaded now so their latency hides behind the mainloop
      const float ws_r = (EPI != EPI_ACC && R < p.N) ? __ldg(p.ws + R) : 0.f;
      const float as_r = (EPI != EPI_ACC && et < NT && tok0 + et < p.M) ? __ldg(p.as + tok0 + et) : 0.f;
      for (int k0 = kb0; k0 < kb1; k0 += p.seg_kb, ++g) {
        if (*abort_flag || !mbar_wait(accf_b(g & 1), (g >> 1) & 1, p.wait_cycles)) { fail(); ok = false; break; }
        drain(g, k0 == kb0);
      }
      if (!ok) break;
      float* asb = as_s + (u & 1) * NT;  // two buffers: unit u+1 writes the other one
      if (et < NT) asb[et] = as_r;
      asm volatile("bar.sync 2, %0;" ::"n"(32 * N_DRAIN_WARPS) : "memory");
      const bool whole = kb0 == 0 && kb1 == nkb;
      if (whole || finish_partial(t)) epilogue(R, tok0 + colh * COLS, ws_r, asb + colh * COLS);
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

// Co-resident CTA pairs of the NT form. The cluster occupancy query counts one pair per
// two SMs for either form; the lean form (NT <= 64) fits two CTAs on an SM, so its count
// is that times the CTAs an SM holds (measured: two lean pairs per two SMs run side by
// side, 64 x 28672 x 4096 in 38 instead of 60 us).
template <int NT>
int max_clusters_t() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device(cache, [] {
    using C = Cfg<NT>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.numAttrs = 0;  // the kernel declares its cluster shape
    int c = 0, dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(k_gemm_tw<EPI_STORE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (cudaOccupancyMaxActiveClusters(&c, k_gemm_tw<EPI_STORE, NT>, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      c = sms / 2;
    }
    // CTAs of this form an SM holds, from its registers and shared memory (the per-SM
    // occupancy query does not take kernels with a compile-time cluster shape)
    cudaFuncAttributes fa{};
    int regs_sm = 0, smem_sm = 0, smem_reserved = 0;
    cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (cudaFuncGetAttributes(&fa, k_gemm_tw<EPI_STORE, NT>) == cudaSuccess)
      for (per_sm = C::CTAS_PER_SM; per_sm > 1; --per_sm)
        if ((long long)fa.numRegs * THREADS * per_sm <= regs_sm &&
            (long long)(C::SMEM_BYTES + fa.sharedSizeBytes + smem_reserved) * per_sm <= smem_sm)
          break;
    cudaGetLastError();
    return std::max(1, c * std::max(1, per_sm));
  });
}
int max_clusters(int nt) {
  return nt == 128 ? max_clusters_t<128>() : (nt == 64 ? max_clusters_t<64>() : max_clusters_t<32>());
}

template <int EPI, int NT>
cudaError_t launch_t(const CUtensorMap& mw, const CUtensorMap& mt, const TcParams& p, int clusters, cudaStream_t s,
                     bool pdl) {
  using C = Cfg<NT>;
  static std::atomic<uint64_t> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    cudaError_t r = cudaFuncSetAttribute(k_gemm_tw<EPI, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (r != cudaSuccess) return r;
    // the register split (setmaxnreg) assumes the launch allocation R_LAUNCH per thread: a drain's
    // increase would wait forever on a smaller pool, so refuse to launch on any other count
    cudaFuncAttributes fa{};
    if ((r = cudaFuncGetAttributes(&fa, k_gemm_tw<EPI, NT>)) != cudaSuccess) return r;
    return fa.numRegs == C::R_LAUNCH ? cudaSuccess : cudaErrorInvalidConfiguration;
  });
  if (e != cudaSuccess) return e;
  return launch_pdl_if(pdl, k_gemm_tw<EPI, NT>, dim3(2 * clusters), dim3(THREADS), (size_t)C::SMEM_BYTES, s, mw, mt,
                       p);
}

template <int EPI>
cudaError_t launch_nt(int nt, const CUtensorMap& mw, const CUtensorMap& mt, const TcParams& p, int clusters,
                      cudaStream_t s, bool pdl) {
  if (nt == 128) return launch_t<EPI, 128>(mw, mt, p, clusters, s, pdl);
  if (nt == 64) return launch_t<EPI, 64>(mw, mt, p, clusters, s, pdl);
  if (nt == 32) return launch_t<EPI, 32>(mw, mt, p, clusters, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_tmap_tw_tokens(CUtensorMap* map, const __half* a16, int rows, int k, int nt) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  if (nt != 128 && nt != 64 && nt != 32) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)(nt / 2)};  // one CTA's token rows
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a16), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_tw_weights(CUtensorMap* map, const int8_t* w, int n, int k) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)k};
  cuuint32_t box[2] = {BK, WM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(w), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Token tile for a chunk of m <= 128 rows: the smallest of 32, 64, 128 that holds it.
int tw_nt(int m) { return m > 64 ? 128 : (m > 32 ? 64 : 32); }

namespace {

// Stream-K plan of one GEMM (ipc == 0: whole tiles round robin).
struct Plan {
  int nt, num_t_tiles, num_tiles, clusters, ipc, max_slots;
  size_t part_elems;
};

Plan plan(int m, int n, int k, bool wide) {
  Plan pl{};
  pl.nt = tw_nt(m);
  const int nkb = k / BK;
  pl.num_t_tiles = (m + pl.nt - 1) / pl.nt;
  pl.num_tiles = pl.num_t_tiles * ((n + 2 * WM - 1) / (2 * WM));
  const int mc = max_clusters(pl.nt);
  if (wide || pl.num_tiles >= mc) {
    pl.clusters = std::min(pl.num_tiles, mc);
    return pl;
  }
  // Fewer tiles than CTA pairs: split the (tile, k-block) space evenly, each pair
  // taking at least min_kb k-blocks to amortise the partial-tile exchange (whose cost
  // grows with the tile: MIN_SK_KB at NT = 128, one exact segment at NT <= 64), and
  // whole tiles when that leaves a pair all of K.
  const long long total = (long long)pl.num_tiles * nkb;
  const int min_kb = pl.nt == 128 ? MIN_SK_KB : MAX_SEG_KB;
  const int ipc = std::max((int)((total + mc - 1) / mc), std::max(MAX_SEG_KB, min_kb));
  if (ipc >= nkb) {
    pl.clusters = std::min(pl.num_tiles, mc);
    return pl;
  }
  pl.ipc = ipc;
  pl.clusters = (int)((total + pl.ipc - 1) / pl.ipc);
  pl.max_slots = (nkb + pl.ipc - 1) / pl.ipc + 1;
  pl.part_elems = (size_t)pl.num_tiles * pl.max_slots * 2 * WM * pl.nt;
  return pl;
}

}  // namespace

void tw_workspace_need(int m, int n, int k, size_t* part_bytes, size_t* counters) {
  const Plan pl = plan(m, n, k, false);
  *part_bytes = pl.part_elems * sizeof(int32_t);
  *counters = pl.ipc ? (size_t)pl.num_tiles * 2 : 0;
}

cudaError_t launch_gemm_tw(int epi, const CUtensorMap& mt, const CUtensorMap& mw, int nt, const float* ws,
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
  p.ws = ws;
  p.as = as;
  p.out = out;
  p.ldo = ldo;
  p.acc_out = acc;
  p.status = status;
  p.rope = rope;
  Plan pl = plan(m, n, k, wide);
  if (m > 128 || pl.nt != nt) return cudaErrorInvalidValue;  // the token map was made for another tile
  p.num_t_tiles = pl.num_t_tiles;
  p.num_tiles = pl.num_tiles;
  if (pl.ipc && wsp.part && wsp.cnt && wsp.part_bytes >= pl.part_elems * sizeof(int32_t) &&
      wsp.counters >= (size_t)pl.num_tiles * 2) {
    p.ipc = pl.ipc;
    p.max_slots = pl.max_slots;
    p.part = wsp.part;
    p.cnt = wsp.cnt;
  } else {
    pl.clusters = std::min(pl.num_tiles, max_clusters(pl.nt));  // no workspace: whole tiles
  }
  switch (epi) {
    case EPI_STORE: return launch_nt<EPI_STORE>(nt, mw, mt, p, pl.clusters, s, pdl);
    case EPI_RESID: return launch_nt<EPI_RESID>(nt, mw, mt, p, pl.clusters, s, pdl);
    case EPI_SWIGLU: return launch_nt<EPI_SWIGLU>(nt, mw, mt, p, pl.clusters, s, pdl);
    case EPI_ACC: return launch_nt<EPI_ACC>(nt, mw, mt, p, pl.clusters, s, pdl);
    case EPI_ROPE:
      if (!rope.table || !rope.q_out || !rope.k_cache || !rope.v_cache || rope.hd % 32 ||
          n != (rope.H + 2 * rope.Hkv) * rope.hd)
        return cudaErrorInvalidValue;
      return launch_nt<EPI_ROPE>(nt, mw, mt, p, pl.clusters, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pp
