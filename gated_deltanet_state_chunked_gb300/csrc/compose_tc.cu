// Tensor-core composition of chunk operators for d_k = d_v = 128.
//
// Method: "LinearKV: One Cached State Suffices for Position-Independent Caching in Hybrid
// LLMs", composition passage (affine chunk operators, exact closed-form composition): the state
// after K chunks is S_K = T_K ... T_1 S_in + sum_j T_K ... T_{j+1} S_local_j in the pages' left
// form, which in the row-major convention of this library (S_out = S_in T^T + S_local) is the
// Horner recursion S_j = S_{j-1} T_j^T + S_local_j, j = 1..K.
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
  volatile int* flag = reinterpret_cast<volatile int*>(sm + L::BARS + 28);

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
    *flag = 0;
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
  // copies of step s into buffer s & 1 (warps 4-7: one T row each, thread 128 also the slice);
  // the buffer's expect_tx was posted before the barrier that precedes this call
  auto issue_loads = [&](int s) {
    if (tid < 128) return;
    const int b = s & 1, r = tid - 128;
    bulk_g2s(sm + L::TB + b * L::TBUF + r * L::TROW, p.T[s] + hoff + (size_t)r * CTD, 512, &bar_ld[b]);
    if (r == 0) bulk_g2s(sm + L::LB + b * 16384, p.Slocal[s] + hoff + (size_t)row0 * CTD, 16384, &bar_ld[b]);
  };
  auto wait_ld = [&](int s) {
    if (!mbar_wait(&bar_ld[s & 1], (uint32_t)((s >> 1) & 1), p.wait_ns)) *flag = 1;
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
    if (!mbar_wait(bar, (uint32_t)(j & 1), p.wait_ns)) *flag = 1;
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
    if (tid == 0 && j + 2 < p.K) mbar_arrive_expect_tx(&bar_ld[j & 1], L::STEP_BYTES);
    __syncthreads();
    if (*flag) break;  // a wait gave up: issue nothing more (every thread reads the flag here)
    if (issuer) issue();
    mma_step = j + 1;
    if (j + 2 < p.K) {
      issue_loads(j + 2);
      issued = j + 2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*flag) {
    // A wait gave up.  What was already issued still runs: let the copies in flight land before
    // the CTA's shared memory is released and the MMAs finish before the TMEM columns are (each
    // wait bounded at the default limit; a wait on a phase that has completed returns at once),
    // then report.
    if (tid == 0) {
      for (int s = 0; s <= issued; ++s) mbar_wait(&bar_ld[s & 1], (uint32_t)((s >> 1) & 1), kWaitNs);
      mbar_wait(bar, (uint32_t)(mma_step & 1), kWaitNs);
      atomicExch(p.status, GDN_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace

bool compose_tc_supported(const ComposeParams& p) { return p.d_k == CTD && p.d_v == CTD && p.K >= 1; }

cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(compose_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)CTLay::ALLOC);
  if (e != cudaSuccess) return e;
  compose_tc_kernel<<<dim3(CTD / CTR, p.h), CTNT, CTLay::ALLOC, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
