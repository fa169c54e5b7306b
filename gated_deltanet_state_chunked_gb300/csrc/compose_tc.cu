// Tensor-core composition of chunk operators for d_k = d_v = 128.
//
// Method: "LinearKV: One Cached State Suffices for Position-Independent Caching in Hybrid
// LLMs", composition passage (affine chunk operators, exact closed-form composition): the state
// after K chunks is S_K = T_K ... T_1 S_in + sum_j T_K ... T_{j+1} S_local_j in the pages' left form,
// which in the row-major convention of this library (S_out = S_in T^T + S_local) is the Horner
// recursion S_j = S_{j-1} T_j^T + S_local_j, j = 1..K.
//
// One CTA per (head, 32-row slice of S), sequential over j.  Transposed, one step is
//   S_j^T (d_k x 32) = T_j (d_k x d_k) S_{j-1}^T + S_local_j^T,
// a tcgen05 MMA with M = 128 (lane = output d_k index), N = 32 (state rows), K = 128:
//   A = T_j split in two, read from TMEM (written there by the threads),
//   B = S_{j-1} rows in shared memory (K-major fp32, 128-byte swizzle).
// fp32 accuracy from three tf32 products per step (split operands, x = hi + lo with hi the
// nearest tf32 value of x and lo = x - hi exact in fp32, read by the MMA as its tf32 part):
// T_hi S_lo + T_lo S_hi + T_hi S_hi, accumulated in fp32 in TMEM.
// A thread issues small MMAs one after another at a fixed cost each, while threads of
// different warps issue side by side: the 48 MMAs of a step are spread over four issuing
// threads (warps 0-3), twelve each, into four accumulators that the epilogue adds.  While they
// run, the threads hold S_local_{j+1} and T_{j+2} loads in flight (fetched as soon as the
// previous values have been used).
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace tcp;

constexpr int CTR = 32;   // state rows per CTA
constexpr int CTNT = 256;  // 8 warps: two per TMEM sub-partition, each owning half the columns
constexpr int CTD = 128;  // d_k = d_v

struct CTLay {
  static constexpr uint32_t SBH = 0;        // S hi: fp32 K-major tile, 32 rows x 128 (4 atoms)
  static constexpr uint32_t SBL = 16384;    // S lo
  static constexpr uint32_t BARS = 32768;
  static constexpr uint32_t TOTAL = BARS + 64;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM columns: tf32(T), T - tf32(T), four accumulators of 32 columns
  static constexpr uint32_t cTH = 0, cTL = 128, cD = 256;
  static constexpr int NACC = 4;
  static constexpr uint32_t TMEM_COLS = 512;
};

__global__ void __launch_bounds__(CTNT, 1) compose_tc_kernel(const ComposeParams p) {
  using L = CTLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 16);
  volatile int* flag = reinterpret_cast<volatile int*>(sm + L::BARS + 24);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, hf = warp >> 2;
  const int h = blockIdx.y, row0 = blockIdx.x * CTR;
  const int m = 32 * quad + lane;  // TMEM lane = d_k index of T's row / of the output column
  const size_t hoff = (size_t)h * CTD * CTD;

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, CTLay::NACC);  // one commit per issuing thread
    mbar_fence_init();
    *flag = 0;
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
  // row m of T_j, columns [64 hf, 64 hf + 64)
  float tr[64];
  auto fetch_T = [&](int j) {
    const float4* src = reinterpret_cast<const float4*>(p.T[j] + hoff + (size_t)m * CTD + 64 * hf);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 v = src[q];
      tr[4 * q] = v.x;
      tr[4 * q + 1] = v.y;
      tr[4 * q + 2] = v.z;
      tr[4 * q + 3] = v.w;
    }
  };
  // S_local_j[row0 + 16 hf + i][m], i < 16: the 16 output rows this thread finishes
  float lr[16];
  auto fetch_L = [&](int j) {
    const float* src = p.Slocal[j] + hoff + (size_t)(row0 + 16 * hf) * CTD + m;
#pragma unroll
    for (int i = 0; i < 16; ++i) lr[i] = src[(size_t)i * CTD];
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  auto store_T = [&]() {  // tr -> tf32(T) and T - tf32(T) columns of this thread's TMEM lane
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32], w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = tf32r(tr[32 * c + i]);
        w[i] = tr[32 * c + i] - v[i];
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

  fetch_T(0);
  store_T();
  tmem_st_wait();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (issuer) issue();
  int issued = 0;  // the last step whose MMAs were issued
  if (p.K > 1) fetch_T(1);
  fetch_L(0);

  for (int j = 0; j < p.K; ++j) {
    // step j's MMAs done: S_j = D + S_local_j
    if (!mbar_wait(bar, (uint32_t)(j & 1), p.wait_ns)) *flag = 1;
    tc_fence_after();
    float d[16], d2[16], d3[16], d4[16];
    tmem_ld16(tmem + lane_base + L::cD + 16 * hf, d);
    tmem_ld16(tmem + lane_base + L::cD + 32 + 16 * hf, d2);
    tmem_ld16(tmem + lane_base + L::cD + 64 + 16 * hf, d3);
    tmem_ld16(tmem + lane_base + L::cD + 96 + 16 * hf, d4);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] += ((d2[i] + d3[i]) + d4[i]) + lr[i];
    if (j + 1 == p.K) {
      float* dst = p.S_out + hoff + (size_t)(row0 + 16 * hf) * CTD + m;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[(size_t)i * CTD] = d[i];
      break;
    }
    fetch_L(j + 1);  // in flight during this step's stores and the next MMAs
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float hi = tf32r(d[i]);
      *reinterpret_cast<float*>(sm + L::SBH + kf32(16 * hf + i, m, CTR)) = hi;
      *reinterpret_cast<float*>(sm + L::SBL + kf32(16 * hf + i, m, CTR)) = d[i] - hi;
    }
    store_T();  // T_{j+1}
    if (j + 2 < p.K) fetch_T(j + 2);
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*flag) break;  // a wait gave up: issue nothing more (every thread reads the flag here)
    if (issuer) issue();
    issued = j + 1;
  }

  tc_fence_before();
  __syncthreads();
  if (*flag) {
    // A wait gave up: the MMAs already issued still write TMEM, so let them finish (their last
    // step's phase, at the default bound) before the columns are released, then report.
    if (tid == 0) {
      mbar_wait(bar, (uint32_t)(issued & 1), kWaitNs);
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
