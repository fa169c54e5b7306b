// Tensor-core composition of chunk operators for d_k = d_v = 128.
//
// Method: "LinearKV: One Cached State Suffices for Position-Independent Caching in Hybrid
// LLMs", composition passage (affine chunk operators, exact closed-form composition): the state
// after K chunks is S_K = T_K ... T_1 S_in + sum_j T_K ... T_{j+1} S_local_j in the pages' left
// form, which in the row-major convention of this library (S_out = S_in T^T + S_local) is the
// Horner recursion S_j = S_{j-1} T_j^T + S_local_j, j = 1..K.
//
// Two kernels: compose_tc_map_kernel (further down) when the T_j sit at one stride in memory,
// fetching each T_j once per head by tensor copies multicast over a cluster; and the kernel
// described here, compose_tc_kernel, for any other pointer array.
//
// One CTA per (head, 32-row slice of S), sequential over j.  Transposed, one step is
//   S_j^T (d_k x 32) = T_j (d_k x d_k) S_{j-1}^T + S_local_j^T,
// a tcgen05 MMA with M = 128 (lane = output d_k index), N = 32 (state rows), K = 128:
//   A = T_j split in two, read from TMEM (written there by the threads),
//   B = S_{j-1} rows in shared memory (K-major fp32, 128-byte swizzle).
// fp32 accuracy from three tf32 products per step (split operands, x = hi + lo with hi the
// nearest tf32 value of x and lo = x - hi exact in fp32, read by the MMA as its tf32 part):
// T_hi S_lo + T_lo S_hi + T_hi S_hi, accumulated in fp32 in TMEM; the 48 MMAs of a step are
// spread over four issuing warps into four accumulators that the epilogue adds.
// Operands stream through shared memory: T_j (one 512-byte row per bulk copy, rows padded to
// 528 bytes so that a warp reading 32 rows touches distinct banks) and the CTA's 16 KB slice of
// S_local_j arrive in one of two buffers, copied by warps 4-7 two steps before they are used, so
// that a step's loads are always in flight behind the previous step's MMAs.
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace tcp;

constexpr int CTR = 32;    // state rows per CTA
constexpr int CTNT = 256;  // 8 warps: two per TMEM sub-partition, each owning half the columns
constexpr int CTD = 128;   // d_k = d_v

struct CTLay {
  static constexpr uint32_t TROW = 528;                 // padded row of a T buffer
  static constexpr uint32_t SBH = 0;                    // S hi: fp32 K-major tile, 32 rows x 128 (4 atoms)
  static constexpr uint32_t SBL = 16384;                // S lo
  static constexpr uint32_t TB = 32768;                 // 2 buffers of T_j (128 rows x 528 B)
  static constexpr uint32_t TBUF = CTD * TROW;          // 67,584
  static constexpr uint32_t LB = TB + 2 * TBUF;         // 2 buffers of the S_local_j slice (32 rows x 512 B)
  static constexpr uint32_t BARS = LB + 2 * 16384;
  static constexpr uint32_t TOTAL = BARS + 64;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  static constexpr uint32_t cTH = 0, cTL = 128, cD = 256;
  static constexpr int NACC = 4;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t STEP_BYTES = CTD * 512 + CTR * 512;
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(LB % 16 == 0 && TB % 16 == 0 && TROW % 16 == 0, "bulk copy alignment");
};

// Advance a shared-memory descriptor's start address by a byte offset (multiple of 16).
__device__ __forceinline__ uint64_t dadd_bytes(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(CTNT, 1) compose_tc_kernel(const ComposeParams p) {
  using L = CTLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BARS);  // MMAs of a step
  uint64_t* bar_ld = bar + 1;                                  // [2] copies of a step
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 24);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, hf = warp >> 2;
  const int h = blockIdx.y, row0 = blockIdx.x * CTR;
  const int m = 32 * quad + lane;
  const size_t hoff = (size_t)h * CTD * CTD;

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, L::NACC);
    mbar_init(&bar_ld[0], 1);
    mbar_init(&bar_ld[1], 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(&bar_ld[0], L::STEP_BYTES);
    if (p.K > 1) mbar_arrive_expect_tx(&bar_ld[1], L::STEP_BYTES);
  }
  // S_0 = S_in (or 0) -> S hi/lo tiles: thread -> row tid / 8, 16 columns
  {
    const int r = tid >> 3, k0 = (tid & 7) * 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.S_in) v = *reinterpret_cast<const float4*>(p.S_in + hoff + (size_t)(row0 + r) * CTD + k0 + 4 * q);
      const float x[4] = {v.x, v.y, v.z, v.w};
      float hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = tf32r(x[e]);
        lo[e] = x[e] - hi[e];
      }
      *reinterpret_cast<float4*>(sm + L::SBH + kf32(r, k0 + 4 * q, CTR)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<float4*>(sm + L::SBL + kf32(r, k0 + 4 * q, CTR)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  int timed_out = 0;  // this thread saw a bounded wait give up
  // copies of step s into buffer s & 1 (warps 4-7: one T row each, thread 128 also the slice);
  // the buffer's expect_tx was posted before the barrier that precedes this call
  auto issue_loads = [&](int s) {
    if (tid < 128) return;
    const int b = s & 1, r = tid - 128;
    bulk_g2s(sm + L::TB + b * L::TBUF + r * L::TROW, p.T[s] + hoff + (size_t)r * CTD, 512, &bar_ld[b]);
    if (r == 0) bulk_g2s(sm + L::LB + b * 16384, p.Slocal[s] + hoff + (size_t)row0 * CTD, 16384, &bar_ld[b]);
  };
  auto wait_ld = [&](int s) {
    if (!mbar_wait(&bar_ld[s & 1], (uint32_t)((s >> 1) & 1), p.wait_ns)) timed_out = 1;
  };
  // row m of T_s, columns [64 hf, 64 hf + 64), from its buffer -> tf32 hi and lo in TMEM
  auto store_T = [&](int s) {
    const unsigned char* src = sm + L::TB + (s & 1) * L::TBUF + m * L::TROW + hf * 256;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32], w[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t = *reinterpret_cast<const float4*>(src + c * 128 + q * 16);
        const float x[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[4 * q + e] = tf32r(x[e]);
          w[4 * q + e] = x[e] - v[4 * q + e];
        }
      }
      tmem_st32(tmem + lane_base + L::cTH + 64 * hf + 32 * c, v);
      tmem_st32(tmem + lane_base + L::cTL + 64 * hf + 32 * c, w);
    }
  };
  const uint64_t dBH = sdesc_sw128(smem_u32(sm + L::SBH), 16, 1024);
  const uint64_t dBL = sdesc_sw128(smem_u32(sm + L::SBL), 16, 1024);
  // MMA n of a step (0..47): pass n / 16 (T_hi S_lo, T_lo S_hi, T_hi S_hi), K step n % 16
  auto mma_n = [&](int n, uint32_t dcol, bool first) {
    constexpr uint32_t id = idesc_tf32(128, CTR);
    const int pass = n >> 4, kk = n & 15;
    const uint32_t a = pass == 1 ? L::cTL : L::cTH;
    const uint64_t b = pass == 0 ? dBL : dBH;
    mma_tf32_ts(tmem + dcol, tmem + a + 8 * kk, b + (uint64_t)((((kk >> 2) * (CTR * 128)) + (kk & 3) * 32) >> 4), id,
                !first);
  };
  // thread 32 w issues MMAs 12 w .. 12 w + 11 into accumulator w (indices fold to constants)
  auto issue = [&]() {
    tc_fence_after();
    const int w = tid >> 5;
    const uint32_t dcol = L::cD + 32 * w;
    switch (w) {
      case 0:
#pragma unroll
        for (int n = 0; n < 12; ++n) mma_n(n, dcol, n == 0);
        break;
      case 1:
#pragma unroll
        for (int n = 12; n < 24; ++n) mma_n(n, dcol, n == 12);
        break;
      case 2:
#pragma unroll
        for (int n = 24; n < 36; ++n) mma_n(n, dcol, n == 24);
        break;
      default:
#pragma unroll
        for (int n = 36; n < 48; ++n) mma_n(n, dcol, n == 36);
        break;
    }
    mma_commit(bar);
  };
  const bool issuer = (tid & 31) == 0 && tid < 32 * L::NACC;

  int issued = p.K > 1 ? 1 : 0;  // last step whose copies were issued
  int mma_step = 0;              // last step whose MMAs were issued
  issue_loads(0);
  if (p.K > 1) issue_loads(1);
  wait_ld(0);
  store_T(0);
  tmem_st_wait();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (issuer) issue();

  for (int j = 0; j < p.K; ++j) {
    // step j's MMAs done: S_j = D + S_local_j
    if (!mbar_wait(bar, (uint32_t)(j & 1), p.wait_ns)) timed_out = 1;
    tc_fence_after();
    float d[16], d2[16], d3[16], d4[16];
    tmem_ld16(tmem + lane_base + L::cD + 16 * hf, d);
    tmem_ld16(tmem + lane_base + L::cD + 32 + 16 * hf, d2);
    tmem_ld16(tmem + lane_base + L::cD + 64 + 16 * hf, d3);
    tmem_ld16(tmem + lane_base + L::cD + 96 + 16 * hf, d4);
    wait_ld(j);  // S_local_j (T_j arrived with it)
    tmem_ld_wait();
    // S_local_j[row0 + 16 hf + i][m]: consecutive m in a warp, consecutive words
    const float* lsl = reinterpret_cast<const float*>(sm + L::LB + (j & 1) * 16384) + (16 * hf) * CTD + m;
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] += ((d2[i] + d3[i]) + d4[i]) + lsl[i * CTD];
    if (j + 1 == p.K) {
      float* dst = p.S_out + hoff + (size_t)(row0 + 16 * hf) * CTD + m;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[(size_t)i * CTD] = d[i];
      break;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float hi = tf32r(d[i]);
      *reinterpret_cast<float*>(sm + L::SBH + kf32(16 * hf + i, m, CTR)) = hi;
      *reinterpret_cast<float*>(sm + L::SBL + kf32(16 * hf + i, m, CTR)) = d[i] - hi;
    }
    wait_ld(j + 1);
    store_T(j + 1);
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    // buffer j & 1 is free once every thread has read S_local_j above (T_j went to TMEM a step ago)
    // (only if this thread saw that phase complete: a pending phase takes no second arrival)
    if (tid == 0 && j + 2 < p.K && !timed_out) mbar_arrive_expect_tx(&bar_ld[j & 1], L::STEP_BYTES);
    // a wait that gave up in any thread stops the loop in every thread (the OR is taken by the barrier)
    if (__syncthreads_or(timed_out)) break;
    if (issuer) issue();
    mma_step = j + 1;
    if (j + 2 < p.K) {
      issue_loads(j + 2);
      issued = j + 2;
    }
  }
  tc_fence_before();
  if (__syncthreads_or(timed_out)) {
    // A wait gave up.  What was already issued still runs: let the copies in flight land before
    // the CTA's shared memory is released and the MMAs finish before the TMEM columns are (each
    // wait bounded at the default limit; a wait on a phase that has completed returns at once),
    // then report.
    if (tid == 0) {
      // the latest issued phase of each copy buffer (an earlier phase of the same buffer has
      // completed, or the later one could not have been issued)
      for (int s = issued > 0 ? issued - 1 : 0; s <= issued; ++s)
        mbar_wait(&bar_ld[s & 1], (uint32_t)((s >> 1) & 1), kWaitNs);
      mbar_wait(bar, (uint32_t)(mma_step & 1), kWaitNs);
      atomicExch(p.status, GDN_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// Composition when the K operators T_1..T_K sit at one stride in memory (one array): every T_j
// row is a row of one 2D view, so a step's T_j arrives by tensor copies (128 rows x 128 B boxes,
// 128-byte swizzle), already in the layout of a K-major tensor-core operand.  The four CTAs of
// a head form a cluster: each fetches one quarter (32 columns) of T_j and multicasts it to all
// four, so T_j leaves L2 once per head instead of four times.  Each thread reads its row of T_j
// (its half of the columns) from the tile once; both operands of the step go to TMEM from there:
//   T_hi [S_lo | S_hi]  one product of N = 64, A = T itself in TMEM (the tensor core reads fp32
//                       as tf32, dropping the low 13 mantissa bits);
//   T_lo S_hi           N = 32, A = T - T_hi in TMEM (exact in fp32), accumulated into the S_hi
//                       half of the same accumulator;
// with K split over two accumulators (added by the epilogue in fp32).  T_lo of step j + 1 is
// written into the other of two TMEM buffers while step j's MMAs run, and T itself into its one
// buffer right after them, so the serial chain per step is the MMAs and the epilogue (D +
// S_local -> the split S tile, T_{j+1} -> TMEM).  The tensor core reads only the S tile from
// shared memory.  T_j sits in one of three shared-memory buffers, refilled as soon as the threads
// have read it, so copies run about three steps ahead; S_local_j is read into registers at the
// top of step j, from L2, where it was prefetched when step j's copies were issued.
//
// Warps 0-7 read T, prepare T_lo and run the epilogue; warp 8 issues the MMAs and owns the
// copies.  Copy protocol: once every thread has read T_s (the barrier before step s's MMAs),
// the CTA posts its own expect_tx for step s + 3 and releases buffer s % 3 by arriving on the
// "free" barrier of that buffer in all four CTAs; it issues its quarter of step s + 3 once its
// own free barrier has all four arrivals.  Every CTA sees the same four arrivals, so a step is
// issued by all four or by none, and a CTA that stops early (a bounded wait gave up) completes
// any step it released before it leaves; a final cluster barrier keeps every CTA alive until
// its partners are done.
// ---------------------------------------------------------------------------------------------
constexpr int kComposeCluster = CTD / CTR;  // CTAs of one head
constexpr int kTBufs = 3;                   // T_j buffers in shared memory
constexpr int kMapThreads = CTNT + 32;      // 8 compute warps and the control warp

struct CMLay {
  static constexpr uint32_t SB = 0;                // [S_lo; S_hi]: fp32 K-major, 64 rows x 4 atoms (8 KB each)
  static constexpr uint32_t TB = 32768;            // kTBufs buffers of T_j: 4 atoms of 128 rows x 128 B (16 KB)
  static constexpr uint32_t TBUF = 65536;
  static constexpr uint32_t BARS = TB + kTBufs * TBUF;
  static constexpr uint32_t TOTAL = BARS + 64;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM: two accumulators of 64 columns (0-31: rows of S_lo, 32-63: rows of S_hi; K steps 0-7
  // and 8-15), T and two T_lo buffers
  static constexpr uint32_t cD = 0, cTH = 128, cTL = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(kComposeCluster == 4, "one box of 32 fp32 columns per CTA of the cluster");
};

__global__ void __cluster_dims__(kComposeCluster, 1, 1) __launch_bounds__(kMapThreads, 1)
    compose_tc_map_kernel(const __grid_constant__ CUtensorMap map_t, const ComposeParams p, int t_rows_per_op) {
  using L = CMLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BARS);  // MMAs of a step
  uint64_t* bar_ld = bar + 1;                                  // [kTBufs] T_j landed in this CTA
  uint64_t* bar_free = bar_ld + kTBufs;                        // [kTBufs] buffer released by all four CTAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_free + kTBufs);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, hf = (warp >> 2) & 1;
  const int h = blockIdx.y, row0 = blockIdx.x * CTR;
  const int rank = (int)cluster_ctarank();  // = blockIdx.x: the quarter of T_j this CTA fetches
  const int m = 32 * quad + lane;           // TMEM lane = d_k index of T's row / of the output column
  const size_t hoff = (size_t)h * CTD * CTD;
  constexpr int kCtl = CTNT / 32;           // the control warp
  constexpr int kLoader = CTNT;             // its lane 0 owns the copies
  const bool ctl = warp == kCtl;
  constexpr uint32_t kTBytes = L::TBUF;     // bytes of T_j landing in each CTA per step

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == kLoader) {
    mbar_init(bar, 1);
    for (int b = 0; b < kTBufs; ++b) {
      mbar_init(&bar_ld[b], 1);
      mbar_init(&bar_free[b], kComposeCluster);
    }
    mbar_fence_init();
    tma_prefetch_desc(&map_t);
    for (int b = 0; b < kTBufs && b < p.K; ++b) mbar_arrive_expect_tx(&bar_ld[b], kTBytes);
  }
  // S_0 = S_in (or 0) -> rows 0-31 (lo) and 32-63 (hi) of the S tile: thread -> row tid / 8, 16 columns
  if (!ctl) {
    const int r = tid >> 3, k0 = (tid & 7) * 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.S_in) v = *reinterpret_cast<const float4*>(p.S_in + hoff + (size_t)(row0 + r) * CTD + k0 + 4 * q);
      const float x[4] = {v.x, v.y, v.z, v.w};
      float hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = tf32r(x[e]);
        lo[e] = x[e] - hi[e];
      }
      *reinterpret_cast<float4*>(sm + L::SB + kf32(r, k0 + 4 * q, 64)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<float4*>(sm + L::SB + kf32(32 + r, k0 + 4 * q, 64)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers are initialised before any copy or arrival reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  int timed_out = 0;  // this thread saw a bounded wait give up
  // this CTA's copies of step s into buffer s % 3 (thread kLoader): its quarter of T_s to all
  // four CTAs (expect_tx already posted for that phase), and its S_local_s rows into L2
  auto issue_loads = [&](int s) {
    const int b = s % kTBufs;
    tma_load_2d_multicast(sm + L::TB + b * L::TBUF + rank * 16384, &map_t, &bar_ld[b], 64 * rank,
                          s * t_rows_per_op + h * CTD, (uint16_t)((1u << kComposeCluster) - 1));
    bulk_prefetch_l2(p.Slocal[s] + hoff + (size_t)row0 * CTD, CTR * 512);
  };
  auto ld_parity = [](int s) { return (uint32_t)((s / kTBufs) & 1); };
  auto wait_ld = [&](int s) {
    if (!mbar_wait(&bar_ld[s % kTBufs], ld_parity(s), p.wait_ns)) timed_out = 1;
  };
  // row m of T_s, columns [64 hf, 64 hf + 64), from the swizzled tile into tr (the 16-byte
  // chunks of a row are XOR-swizzled by its index: a warp's rows hit distinct banks), and
  // T - T_hi into T_lo buffer s & 1
  float tr[64];
  auto load_T = [&](int s) {
    const unsigned char* tile = sm + L::TB + (s % kTBufs) * L::TBUF + (uint32_t)m * 128u;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int a = 2 * hf + c;  // atom = 32 columns
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t = *reinterpret_cast<const float4*>(tile + a * 16384 + (((uint32_t)q ^ (m & 7u)) << 4));
        tr[32 * c + 4 * q] = t.x;
        tr[32 * c + 4 * q + 1] = t.y;
        tr[32 * c + 4 * q + 2] = t.z;
        tr[32 * c + 4 * q + 3] = t.w;
      }
      float w[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = tr[32 * c + e];
        w[e] = x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
      }
      tmem_st32(tmem + lane_base + L::cTL + 128 * (s & 1) + 32 * a, w);
    }
  };
  // T itself (the row held in tr) into the T buffer, once the MMAs reading the previous T are done
  auto store_T = [&]() {
    tmem_st32(tmem + lane_base + L::cTH + 64 * hf, *reinterpret_cast<const float(*)[32]>(tr));
    tmem_st32(tmem + lane_base + L::cTH + 64 * hf + 32, *reinterpret_cast<const float(*)[32]>(tr + 32));
  };
  const uint64_t dS = sdesc_sw128(smem_u32(sm + L::SB), 16, 1024);          // [S_lo; S_hi], N = 64
  const uint64_t dShi = sdesc_sw128(smem_u32(sm + L::SB + 4096), 16, 1024);  // S_hi rows, N = 32
  // step s's 32 MMAs, one issuing thread of the control warp, in K order; each T_lo S_hi term
  // follows the T_hi [S_lo | S_hi] term of its K step, the first of which initialises its accumulator
  auto issue = [&](int s) {
    tc_fence_after();
    constexpr uint32_t id64 = idesc_tf32(128, 64);
    constexpr uint32_t id32 = idesc_tf32(128, CTR);
    const uint32_t tl = tmem + L::cTL + 128 * (s & 1);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t kb = (kk >> 2) * 8192 + (kk & 3) * 32;  // K step in the S tile (64-row atoms)
      const uint32_t dc = tmem + L::cD + 64 * (kk >> 3);
      if (elect_one()) {
        mma_tf32_ts(dc, tmem + L::cTH + 8 * kk, dadd_bytes(dS, kb), id64, (kk & 7) > 0);
        mma_tf32_ts(dc + 32, tl + 8 * kk, dadd_bytes(dShi, kb), id32, true);
      }
    }
    if (elect_one()) mma_commit(bar);
    __syncwarp();
  };

  // thread kLoader's record: last step whose copies it issued, last step it released a buffer for
  int issued = (p.K < kTBufs ? p.K : kTBufs) - 1, released = issued;
  int mma_step = 0;  // last step whose MMAs were issued
  // thread kLoader, once every thread has read T_{s - 3}: release its buffer for step s (after
  // seeing step s - 3's copies complete) and, once all four CTAs have, issue step s's copies
  auto refill = [&](int s) {
    const int b = s % kTBufs;
    if (timed_out || !mbar_wait(&bar_ld[b], ld_parity(s - kTBufs), p.wait_ns)) {
      timed_out = 1;
      return;
    }
    mbar_arrive_expect_tx(&bar_ld[b], kTBytes);
#pragma unroll
    for (int c = 0; c < kComposeCluster; ++c) mbar_arrive_remote_relaxed(&bar_free[b], (uint32_t)c);
    released = s;
    if (mbar_wait_cluster(&bar_free[b], ld_parity(s - kTBufs), p.wait_ns)) {
      issue_loads(s);
      issued = s;
    } else {
      timed_out = 1;  // the loop stops at a later barrier (the copy waits give up)
    }
  };
  if (ctl) {
    if (tid == kLoader)
      for (int s = 0; s <= issued; ++s) issue_loads(s);
    __syncwarp();
  } else {
    wait_ld(0);
    load_T(0);
    store_T();
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (ctl) {
    issue(0);
    if (tid == kLoader && kTBufs < p.K) refill(kTBufs);  // T_0 has been read
    __syncwarp();
    // control warp: issue each step's MMAs once the compute warps have written its S tile, T and
    // T_lo; then refill the buffer of the T they read before that barrier
    for (int j = 0; j + 1 < p.K; ++j) {
      if (__syncthreads_or(timed_out)) break;
      issue(j + 1);
      mma_step = j + 1;
      if (tid == kLoader && j + 1 + kTBufs < p.K) refill(j + 1 + kTBufs);
      __syncwarp();
    }
  } else {
    for (int j = 0; j < p.K; ++j) {
      // S_local_j[row0 + 16 hf + i][m] (consecutive m in a warp: coalesced), used by the epilogue
      float sl[16];
      {
        const float* src = p.Slocal[j] + hoff + (size_t)(row0 + 16 * hf) * CTD + m;
#pragma unroll
        for (int i = 0; i < 16; ++i) sl[i] = __ldg(src + (size_t)i * CTD);
      }
      // while step j's MMAs run: T_{j+1} into registers and its T_lo into the other TMEM buffer
      // (step j - 1's MMAs, the last readers of that buffer, completed before the previous barrier)
      if (j + 1 < p.K) {
        wait_ld(j + 1);
        load_T(j + 1);
      }
      // step j's MMAs done: S_j = D + S_local_j
      if (!mbar_wait(bar, (uint32_t)(j & 1), p.wait_ns)) timed_out = 1;
      tc_fence_after();
      float d[16], x[16], y[16];
      tmem_ld16(tmem + lane_base + L::cD + 16 * hf, d);
      tmem_ld16(tmem + lane_base + L::cD + 32 + 16 * hf, x);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) d[i] += x[i];
      tmem_ld16(tmem + lane_base + L::cD + 64 + 16 * hf, x);
      tmem_ld16(tmem + lane_base + L::cD + 96 + 16 * hf, y);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) d[i] += (x[i] + y[i]) + sl[i];
      if (j + 1 == p.K) {
        float* dst = p.S_out + hoff + (size_t)(row0 + 16 * hf) * CTD + m;
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[(size_t)i * CTD] = d[i];
        break;
      }
      store_T();  // step j's MMAs, the readers of the T buffer, are done
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float hi = tf32r(d[i]);
        *reinterpret_cast<float*>(sm + L::SB + kf32(16 * hf + i, m, 64)) = d[i] - hi;
        *reinterpret_cast<float*>(sm + L::SB + kf32(32 + 16 * hf + i, m, 64)) = hi;
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      // a wait that gave up in any thread stops the loop in every thread (the OR is taken by the barrier)
      if (__syncthreads_or(timed_out)) break;
    }
  }

  tc_fence_before();
  if (__syncthreads_or(timed_out)) {
    // A wait gave up.  Complete a step this CTA released but has not issued (its partners issue
    // theirs when they see the same four releases), let the copies into this CTA land and the
    // MMAs finish (each wait bounded at the default limit), then report.
    if (tid == kLoader) {
      if (released > issued) {
        const int s = released;
        if (mbar_wait_cluster(&bar_free[s % kTBufs], ld_parity(s - kTBufs), kWaitNs)) {
          issue_loads(s);
          issued = s;
        }
      }
      // the latest phase of each buffer (its earlier phases completed before it was reissued)
      for (int s = issued >= kTBufs - 1 ? issued - (kTBufs - 1) : 0; s <= issued; ++s)
        mbar_wait(&bar_ld[s % kTBufs], ld_parity(s), kWaitNs);
    }
    if (tid == kLoader) {
      mbar_wait(bar, (uint32_t)(mma_step & 1), kWaitNs);
      atomicExch(p.status, GDN_ERR_TIMEOUT);
    }
    __syncthreads();
  }
  // no CTA leaves while a partner may still write into it or arrive on its barriers
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace

bool compose_tc_supported(const ComposeParams& p) { return p.d_k == CTD && p.d_v == CTD && p.K >= 1; }

cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t stream) {
  // One 2D view covers every T_j when they sit at one non-negative stride that is a whole number
  // of 512-byte rows (one array of operators); otherwise each step's rows are copied one by one.
  const char* t0 = reinterpret_cast<const char*>(p.T[0]);
  const ptrdiff_t stride = p.K > 1 ? reinterpret_cast<const char*>(p.T[1]) - t0 : 0;
  bool uniform = stride >= 0 && stride % 512 == 0;
  for (int j = 2; uniform && j < p.K; ++j) uniform = reinterpret_cast<const char*>(p.T[j]) == t0 + j * stride;
  const uint64_t rows_per_op = (uint64_t)stride / 512;
  const uint64_t rows = (uint64_t)(p.K - 1) * rows_per_op + (uint64_t)p.h * CTD;
  CUtensorMap map;
  if (uniform && rows < (1ull << 31) && make_map(&map, t0, rows, 2 * CTD, CTD)) {
    cudaError_t e = cudaFuncSetAttribute(compose_tc_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)CMLay::ALLOC);
    if (e != cudaSuccess) return e;
    compose_tc_map_kernel<<<dim3(CTD / CTR, p.h), kMapThreads, CMLay::ALLOC, stream>>>(map, p, (int)rows_per_op);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(compose_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)CTLay::ALLOC);
  if (e != cudaSuccess) return e;
  compose_tc_kernel<<<dim3(CTD / CTR, p.h), CTNT, CTLay::ALLOC, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
