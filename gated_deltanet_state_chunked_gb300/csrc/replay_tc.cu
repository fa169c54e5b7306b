// Tensor-core (tcgen05 + TMEM + TMA) chunked scan for bf16 inputs, d_k = d_v = 128.
//
// Method: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix
// Caching for Hybrid LLMs", section 2 Eq. (1) and section 3 Eq. (2), evaluated
// chunk by chunk (C = 64 tokens).  With normalised keys k^_t = rk_t k_t,
// queries q^_t = scale rq_t q_t, inclusive gate sums G_t, gamma_t = exp(G_t)
// and the chunk's entering state S0 (d_v x d_k):
//   A_ts = beta_t exp(G_t - G_s) k^_t.k^_s  (s < t),   M = (I + A)^{-1}
//   U~   = M diag(beta) V                     W = M diag(beta gamma rk) K
//   U    = U~ - W S0^T                        (the corrected values)
//   S    = gamma_C S0 + K^T diag(rk exp(G_C - G_s)) U     (carried in fp32)
//   O    = diag(gamma) Q^ S0^T + P U,   P_ts = exp(G_t - G_s) q^_t.k^_s (s <= t)
//
// Two kernels:
//  * chunk_prep_kernel -- one CTA per (chunk, key head), all chunks of all tails
//    in parallel: K K^T on tcgen05, the gated A, and M = (I + A)^{-1} on CUDA
//    cores (16x16 diagonal blocks by substitution, then block merges), written
//    with beta, G and rk to a per-(chunk, v-head) record in scratch memory.
//  * chunk_scan_kernel -- one CTA per R-row slice (R = 32 or 64 rows of d_v) of
//    one (tail, v-head) state, walking the tail's chunks.  Per chunk:
//      Q K^T              bf16 (exact inputs)                          M=64  N=64
//      [Mw_hi|Mw_lo][K;K] bf16 hi/lo split of the computed factor        M=64  N=128 K=128
//      [Mb_hi|Mb_lo][V;V] same                                           M=64  N=R   K=128
//      W S0^T             tf32 (operands rounded to nearest)             M=64  N=R   K=128
//      Q [S0_hi|S0_lo]^T  bf16 split of the state                        M=64  N=R   K=256
//      [K^T|K^T][U^hi;U^lo] bf16 split of the scaled U                   M=128 N=R   K=128
//      P U                tf32                                           M=64  N=R   K=64
//    all accumulated in fp32 in TMEM; the state slice stays in fp32 registers.
// Padded tokens past a tail's end get beta = g = 0 (identity transitions).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace tcp;

constexpr int NT = 256;

// ---------------------------------------------------------------------------------------------
// prep kernel
// ---------------------------------------------------------------------------------------------
constexpr int MST = 68;  // row stride (floats) of the 64x64 fp32 work matrices
struct PrepLay {
  static constexpr uint32_t KT = 0;                      // bf16 K tile: 2 d_k atoms x (64 rows x 128 B)
  static constexpr uint32_t AMAT = 16384;                // fp32 64 x 68
  static constexpr uint32_t MMAT = AMAT + 64 * MST * 4;  // fp32 64 x 68
  static constexpr uint32_t GATE = MMAT + 64 * MST * 4;  // beta[64], G2[64], rk[64]
  static constexpr uint32_t BARS = GATE + 768;           // 2 mbarriers, TMEM slot, scratch ints
  static constexpr uint32_t TOTAL = BARS + 128;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
};

struct PrepParams {
  const float* g;
  const float* beta;
  const int32_t* cu;
  unsigned char* rec;  // records [chunk][h_v]
  int* status;
  int n_seqs, total_tokens, h_k, h_v, l2norm;
};

// M = (I + A)^{-1} for a 64x64 strictly lower A (stride MST).  256 threads.
// A's strictly upper blocks are used as scratch (overwritten).
__device__ void invert_unit_lower(float* A, float* M) {
  const int tid = threadIdx.x;
  if (tid < 64) {  // diagonal blocks by forward substitution, one column per thread
    const int b = tid >> 4, j = tid & 15;
    const float* Ab = A + (16 * b) * MST + 16 * b;
    float m[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float a0 = (t == j) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
      for (int s = 0; s < t; s += 2) {
        a0 = fmaf(-Ab[t * MST + s], m[s], a0);
        if (s + 1 < t) a1 = fmaf(-Ab[t * MST + s + 1], m[s + 1], a1);
      }
      m[t] = a0 + a1;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) M[(16 * b + t) * MST + 16 * b + j] = m[t];
  } else {
    for (int i = tid - 64; i < 64 * 64; i += NT - 64) {
      const int t = i >> 6, s = i & 63;
      if ((s >> 4) > (t >> 4)) M[t * MST + s] = 0.f;
    }
  }
  __syncthreads();
  // At_ik = M_ii A_ik for the six strictly lower blocks, kept in A's block (k, i)
  for (int task = tid; task < 384; task += NT) {
    const int blk = task >> 6, r = (task >> 2) & 15, cq = (task & 3) * 4;
    const int i = blk < 1 ? 1 : (blk < 3 ? 2 : 3);
    const int k = blk < 1 ? 0 : (blk < 3 ? blk - 1 : blk - 3);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float m = M[(16 * i + r) * MST + 16 * i + u];
      const float4 a = *reinterpret_cast<const float4*>(A + (16 * i + u) * MST + 16 * k + cq);
      acc.x = fmaf(m, a.x, acc.x); acc.y = fmaf(m, a.y, acc.y);
      acc.z = fmaf(m, a.z, acc.z); acc.w = fmaf(m, a.w, acc.w);
    }
    *reinterpret_cast<float4*>(A + (16 * k + r) * MST + 16 * i + cq) = acc;
  }
  __syncthreads();
  // M_ij = -sum_{k=j}^{i-1} At_ik M_kj, block diagonals d = 1, 2, 3
#pragma unroll
  for (int d = 1; d < 4; ++d) {
    for (int task = tid; task < (4 - d) * 64; task += NT) {
      const int i = d + (task >> 6), j = i - d, r = (task >> 2) & 15, cq = (task & 3) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = j; k < i; ++k) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float a = A[(16 * k + r) * MST + 16 * i + u];
          const float4 m = *reinterpret_cast<const float4*>(M + (16 * k + u) * MST + 16 * j + cq);
          acc.x = fmaf(a, m.x, acc.x); acc.y = fmaf(a, m.y, acc.y);
          acc.z = fmaf(a, m.z, acc.z); acc.w = fmaf(a, m.w, acc.w);
        }
      }
      *reinterpret_cast<float4*>(M + (16 * i + r) * MST + 16 * j + cq) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(NT, 4) chunk_prep_kernel(const __grid_constant__ CUtensorMap map_k, PrepParams p) {
  using L = PrepLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* amat = reinterpret_cast<float*>(sm + L::AMAT);
  float* mmat = reinterpret_cast<float*>(sm + L::MMAT);
  float* gBeta = reinterpret_cast<float*>(sm + L::GATE);
  float* gG2 = gBeta + 64;
  float* gRk = gBeta + 128;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 16);
  int* scratch = reinterpret_cast<int*>(sm + L::BARS + 32);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, half = warp >> 2;
  const int gc = blockIdx.x, hk = blockIdx.y;
  const ChunkInfo ci = chunk_info(p.cu, p.n_seqs, p.total_tokens, -1, gc, scratch);
  if (gc >= ci.total || ci.gc_seq < 0) return;
  const int t0 = p.cu[ci.gc_seq] + ci.gc_idx * C;
  const int n = min(C, p.cu[ci.gc_seq + 1] - t0);
  const int G = p.h_v / p.h_k;

  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(bar_tma, 16384);
    tma_load_2d(sm + L::KT, &map_k, bar_tma, hk * DK, t0);
    tma_load_2d(sm + L::KT + 8192, &map_k, bar_tma, hk * DK + 64, t0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = mbar_wait(bar_tma, 0, kWaitNs);
  if (tid == 0) {
    const uint32_t k0 = smem_u32(sm + L::KT);
    constexpr uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint64_t d = sdesc_sw128(k0 + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024);
      mma_bf16(tmem, d, d, id, j > 0);
    }
    mma_commit(bar_mma);
  }
  if (tid < 128) {  // key norms from the bf16 tile (row sums need no un-swizzling)
    const int row = tid >> 1, atom = tid & 1;
    const uint4* src = reinterpret_cast<const uint4*>(sm + L::KT + atom * 8192 + row * 128);
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 u = src[c];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    if (atom == 0) gRk[row] = p.l2norm ? 1.f / sqrtf(ss + 1e-6f) : 1.f;
  }
  ok = mbar_wait(bar_mma, 0, kWaitNs) && ok;
  tc_fence_after();
  float kk[32];  // this thread's 32 columns of K K^T (M=64 layout: rows 16*quad + lane, lane < 16)
  tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + half * 32, kk);
  tmem_ld_wait();
  if (!ok && tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);

  for (int j = 0; j < G; ++j) {
    const int h = hk * G + j;
    __syncthreads();
    if (warp == 0) {  // gates: beta, inclusive gate sums (log2 units); padding gets 0
      float ga = lane < n ? p.g[(size_t)(t0 + lane) * p.h_v + h] : 0.f;
      float gb = lane + 32 < n ? p.g[(size_t)(t0 + lane + 32) * p.h_v + h] : 0.f;
      gBeta[lane] = lane < n ? p.beta[(size_t)(t0 + lane) * p.h_v + h] : 0.f;
      gBeta[lane + 32] = lane + 32 < n ? p.beta[(size_t)(t0 + lane + 32) * p.h_v + h] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float xa = __shfl_up_sync(0xffffffffu, ga, o);
        const float xb = __shfl_up_sync(0xffffffffu, gb, o);
        if (lane >= o) { ga += xa; gb += xb; }
      }
      gb += __shfl_sync(0xffffffffu, ga, 31);
      gG2[lane] = ga * kLog2e;
      gG2[lane + 32] = gb * kLog2e;
    }
    __syncthreads();
    if (lane < 16) {
      const int t = 16 * quad + lane;
      const float bt = gBeta[t] * gRk[t], gt = gG2[t];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int s = half * 32 + i;
        amat[t * MST + s] = s < t ? bt * exp2f(gt - gG2[s]) * gRk[s] * kk[i] : 0.f;
      }
    }
    __syncthreads();
    invert_unit_lower(amat, mmat);
    // record
    unsigned char* rec = p.rec + ((size_t)gc * p.h_v + h) * kRecBytes;
    for (int i = tid; i < 64 * 16; i += NT) {
      const int t = i >> 4, q4 = (i & 15) * 4;
      *reinterpret_cast<float4*>(rec + kRecM + (t * 64 + q4) * 4) = *reinterpret_cast<const float4*>(mmat + t * MST + q4);
    }
    if (tid < 64) {
      reinterpret_cast<float*>(rec + kRecBeta)[tid] = gBeta[tid];
      reinterpret_cast<float*>(rec + kRecG2)[tid] = gG2[tid];
      reinterpret_cast<float*>(rec + kRecRk)[tid] = gRk[tid];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------------------------------------
// scan kernel
// ---------------------------------------------------------------------------------------------
template <int R>
struct ScanLay {
  static constexpr uint32_t KQ = 0;                 // bf16 [K;Q]: 2 d_k atoms x (128 rows x 128 B)
  static constexpr uint32_t VT = KQ + 32768;        // bf16 V atom: 64 tokens x 128 B
  static constexpr uint32_t REC = VT + 8192;        // the chunk's record (M, beta, G2, rk)
  static constexpr uint32_t XR = REC + kRecBytes;   // 32 KB, three lives per chunk:
  static constexpr uint32_t MB = XR;                //   bf16 [Mb_hi|Mb_lo] (64 rows x 2 atoms)
  static constexpr uint32_t MW = XR + 16384;        //   bf16 [Mw_hi|Mw_lo]
  static constexpr uint32_t WQ = XR;                //   fp32 W (64 rows x 4 atoms), tf32-rounded
  static constexpr uint32_t UH = XR;                //   bf16 [U^hi;U^lo] MN-major (128 token rows x 128 B)
  static constexpr uint32_t UT = XR + 16384;        //   fp32 U^T (R rows x 2 atoms)
  static constexpr uint32_t S32 = XR + 32768;       // fp32 state slice (R rows x 4 atoms), tf32-rounded
  static constexpr uint32_t SHL = S32 + R * 512;    // bf16 state hi (R rows x 2 atoms), then lo
  static constexpr uint32_t P32 = SHL + R * 512;    // fp32 P (64 rows x 2 atoms)
  static constexpr uint32_t GATE = P32 + 16384;     // gamma[64], wsc[64], rq[64], G2-scratch
  static constexpr uint32_t BARS = GATE + 1024;
  static constexpr uint32_t TOTAL = BARS + 128;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM columns
  static constexpr uint32_t cQK = 0, cW = 64, cU = 192, cD1w = 192 + R, cD1q = 192 + 2 * R, cD2 = 192 + 3 * R,
                            cPU = 192 + 4 * R;
  static_assert(192 + 5 * R <= 512, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(XR % 1024 == 0 && S32 % 1024 == 0 && P32 % 1024 == 0, "tile alignment");
};

struct ScanParams {
  const int32_t* cu;
  const float* S0;
  const unsigned char* rec;
  __nv_bfloat16* O;
  float* S_out;
  int* status;
  int n_seqs, total_tokens, h_k, h_v;
  int l2norm, write_O;
  float scale;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[16]) { tmem_ld16(taddr, v); }

template <int R>
__global__ void __launch_bounds__(NT, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, ScanParams p) {
  using L = ScanLay<R>;
  constexpr int HALF = R / 2;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const float* rM = reinterpret_cast<const float*>(sm + L::REC + kRecM);
  const float* rBeta = reinterpret_cast<const float*>(sm + L::REC + kRecBeta);
  const float* rG2 = reinterpret_cast<const float*>(sm + L::REC + kRecG2);
  const float* rRk = reinterpret_cast<const float*>(sm + L::REC + kRecRk);
  float* gGam = reinterpret_cast<float*>(sm + L::GATE);
  float* gWsc = gGam + 64;
  float* gRq = gGam + 128;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_qk = bar_tma + 1;
  uint64_t* bar_mma = bar_tma + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 24);
  int* abort_flag = reinterpret_cast<int*>(sm + L::BARS + 28);
  int* scratch = reinterpret_cast<int*>(sm + L::BARS + 64);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int slice = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int row0 = slice * R;
  const int hk = h / (p.h_v / p.h_k);

  const int t_begin = p.cu[seq], t_end = p.cu[seq + 1];
  if (t_begin < 0 || t_end < t_begin || t_end > p.total_tokens) {
    if (tid == 0) atomicExch(p.status, GDN_ERR_SHAPE);
    return;
  }
  const ChunkInfo ci = chunk_info(p.cu, p.n_seqs, p.total_tokens, seq, -1, scratch);

  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_qk, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    *abort_flag = 0;
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
  }

  // entering state: thread owns d = 32*quad + lane and columns [half*HALF, +HALF), fp32 registers
  const int dcol = 32 * quad + lane;
  float sreg[HALF];
  const size_t sbase = ((size_t)seq * p.h_v + h) * DV * DK;
#pragma unroll
  for (int i = 0; i < HALF; ++i) {
    const int c = half * HALF + i;
    const float s = p.S0 ? p.S0[sbase + (size_t)(row0 + c) * DK + dcol] : 0.f;
    sreg[i] = s;
    *reinterpret_cast<float*>(sm + L::S32 + kf32(c, dcol, R)) = tf32r(s);
    const __nv_bfloat16 hi = __float2bfloat16_rn(s);
    *reinterpret_cast<__nv_bfloat16*>(sm + L::SHL + kbf16(c, dcol, R)) = hi;
    *reinterpret_cast<__nv_bfloat16*>(sm + L::SHL + R * 256 + kbf16(c, dcol, R)) =
        __float2bfloat16_rn(s - __bfloat162float(hi));
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t sKQ = smem_u32(sm + L::KQ), sVT = smem_u32(sm + L::VT), sXR = smem_u32(sm + L::XR);
  const uint32_t sS32 = smem_u32(sm + L::S32), sSHL = smem_u32(sm + L::SHL), sP32 = smem_u32(sm + L::P32);
  const uint32_t vcoloff = (uint32_t)(row0 & 63) * 2u;
  uint32_t tma_ph = 0, qk_ph = 0, mma_ph = 0;
  bool ok = true;
  int gcur = ci.first;

  for (int t0 = t_begin; t0 < t_end; t0 += C, ++gcur) {
    const int n = min(C, t_end - t0);
    // ---------------------------------------------------------------- loads
    if (tid == 0) {
      fence_async_smem();
      mbar_arrive_expect_tx(bar_tma, 32768 + 8192 + kRecBytes);
      for (int a = 0; a < 2; ++a) {
        tma_load_2d(sm + L::KQ + a * 16384, &map_k, bar_tma, hk * DK + a * 64, t0);
        tma_load_2d(sm + L::KQ + a * 16384 + 8192, &map_q, bar_tma, hk * DK + a * 64, t0);
      }
      tma_load_2d(sm + L::VT, &map_v, bar_tma, h * DV + (row0 & ~63), t0);
      bulk_load(sm + L::REC, p.rec + ((size_t)gcur * p.h_v + h) * kRecBytes, kRecBytes, bar_tma);
    }
    if (!mbar_wait(bar_tma, tma_ph & 1, kWaitNs)) *abort_flag = 1;
    ++tma_ph;
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    // ---------------------------------------------------------------- Q K^T (outputs only)
    if (tid == 0 && p.write_O) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t off = (j >> 2) * 16384 + (j & 3) * 32;
        mma_bf16(tmem + L::cQK, sdesc_sw128(sKQ + 8192 + off, 16, 1024), sdesc_sw128(sKQ + off, 16, 1024), id, j > 0);
      }
      mma_commit(bar_qk);
    }
    // gates, query norms, and the bf16 hi|lo factors Mb = M diag(beta), Mw = M diag(beta gamma rk)
    if (tid < 64) {
      const float l = rG2[63];
      gGam[tid] = exp2f(rG2[tid]);
      gWsc[tid] = exp2f(l - rG2[tid]) * rRk[tid];
    } else if (tid < 192 && p.write_O) {
      const int row = (tid - 64) >> 1, atom = tid & 1;
      const uint4* src = reinterpret_cast<const uint4*>(sm + L::KQ + atom * 16384 + 8192 + row * 128);
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 u = src[c];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (atom == 0) gRq[row] = (p.l2norm ? 1.f / sqrtf(ss + 1e-6f) : 1.f) * p.scale;
    }
    {
      const int t = tid >> 2, s0 = (tid & 3) * 16;
      __align__(16) __nv_bfloat16 bh[16], bl[16], wh[16], wl[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int s = s0 + i;
        const float mb = rM[t * 64 + s] * rBeta[s];
        const float mw = mb * exp2f(rG2[s]) * rRk[s];
        bh[i] = __float2bfloat16_rn(mb);
        bl[i] = __float2bfloat16_rn(mb - __bfloat162float(bh[i]));
        wh[i] = __float2bfloat16_rn(mw);
        wl[i] = __float2bfloat16_rn(mw - __bfloat162float(wh[i]));
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int s = s0 + 8 * c;
        *reinterpret_cast<uint4*>(sm + L::MB + kbf16(t, s, 64)) = reinterpret_cast<const uint4*>(bh)[c];
        *reinterpret_cast<uint4*>(sm + L::MB + kbf16(t, 64 + s, 64)) = reinterpret_cast<const uint4*>(bl)[c];
        *reinterpret_cast<uint4*>(sm + L::MW + kbf16(t, s, 64)) = reinterpret_cast<const uint4*>(wh)[c];
        *reinterpret_cast<uint4*>(sm + L::MW + kbf16(t, 64 + s, 64)) = reinterpret_cast<const uint4*>(wl)[c];
      }
    }
    fence_async_smem();
    __syncthreads();
    // ---------------------------------------------------------------- W = Mw K, U~ = Mb V
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idW = idesc_bf16(64, 128, false, true);
      constexpr uint32_t idU = idesc_bf16(64, R, false, true);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t kb = (j >> 2) * 8192 + (j & 3) * 32;
        const uint32_t rows = (j & 3) * 16 * 128;
        mma_bf16(tmem + L::cW, sdesc_sw128(sXR + 16384 + kb, 16, 1024), sdesc_sw128(sKQ + rows, 16384, 1024), idW,
                 j > 0);
        mma_bf16(tmem + L::cU, sdesc_sw128(sXR + kb, 16, 1024), sdesc_sw128(sVT + vcoloff + rows, 8192, 1024), idU,
                 j > 0);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    // ---------------------------------------------------------------- P (outputs only)
    if (p.write_O) {
      if (!mbar_wait(bar_qk, qk_ph & 1, kWaitNs)) *abort_flag = 1;
      ++qk_ph;
      tc_fence_after();
      float v[32];
      ld_cols(tmem + lane_base + L::cQK + half * 32, v);
      tmem_ld_wait();
      if (lane < 16) {
        const int t = 16 * quad + lane;
        const float qt = gRq[t], gt = rG2[t];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = half * 32 + i + e;
            x[e] = s <= t ? tf32r(qt * exp2f(gt - rG2[s]) * rRk[s] * v[i + e]) : 0.f;
          }
          *reinterpret_cast<float4*>(sm + L::P32 + kf32(t, half * 32 + i, 64)) = make_float4(x[0], x[1], x[2], x[3]);
        }
      }
    }
    if (!mbar_wait(bar_mma, mma_ph & 1, kWaitNs)) *abort_flag = 1;
    ++mma_ph;
    tc_fence_after();
    // ---------------------------------------------------------------- W -> tf32 tile
    {
      const int t = 16 * quad + lane;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
        const int d0 = half * 64 + cc * 32;
        ld_cols(tmem + lane_base + L::cW + d0, v);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(sm + L::WQ + kf32(t, d0 + i, 64)) =
                make_float4(tf32r(v[i]), tf32r(v[i + 1]), tf32r(v[i + 2]), tf32r(v[i + 3]));
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------------------------------------------------------- W S0^T (tf32), Q [S0_hi|S0_lo]^T (bf16)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idw = idesc_tf32(64, R);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint64_t a = sdesc_sw128(sXR + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024);
        const uint64_t b = sdesc_sw128(sS32 + (j >> 2) * (R * 128) + (j & 3) * 32, 16, 1024);
        mma_tf32(tmem + L::cD1w, a, b, idw, j > 0);
      }
      if (p.write_O) {
        constexpr uint32_t idq = idesc_bf16(64, R, false, false);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t kk = j & 7;  // K step inside d_k; j >= 8 uses the lo half of the state
          const uint64_t a = sdesc_sw128(sKQ + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sSHL + (j >> 3) * (R * 256) + (kk >> 2) * (R * 128) + (kk & 3) * 32, 16, 1024);
          mma_bf16(tmem + L::cD1q, a, b, idq, j > 0);
        }
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    if (!mbar_wait(bar_mma, mma_ph & 1, kWaitNs)) *abort_flag = 1;
    ++mma_ph;
    tc_fence_after();
    // ---------------------------------------------------------------- U = U~ - W S0^T; U^ hi/lo (MN-major), U^T (tf32)
    {
      const int t = 16 * quad + lane;
      float ut[HALF], dw[HALF];
      ld_cols(tmem + lane_base + L::cU + half * HALF, ut);
      ld_cols(tmem + lane_base + L::cD1w + half * HALF, dw);
      tmem_ld_wait();
      if (lane < 16) {
        const float sc = gWsc[t];
        __align__(16) __nv_bfloat16 hi[HALF], lo[HALF];
#pragma unroll
        for (int i = 0; i < HALF; ++i) {
          const float u = ut[i] - dw[i];
          const int c = half * HALF + i;
          *reinterpret_cast<float*>(sm + L::UT + kf32(c, t, R)) = tf32r(u);
          const float uh = u * sc;
          hi[i] = __float2bfloat16_rn(uh);
          lo[i] = __float2bfloat16_rn(uh - __bfloat162float(hi[i]));
        }
#pragma unroll
        for (int i = 0; i < HALF; i += 8) {
          const int c = half * HALF + i;
          *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(c, t, 128)) = *reinterpret_cast<const uint4*>(hi + i);
          *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(c, 64 + t, 128)) = *reinterpret_cast<const uint4*>(lo + i);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------------------------------------------------------- K^T U^ (state), P U (outputs)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t id2 = idesc_bf16(128, R, true, true);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mma_bf16(tmem + L::cD2, sdesc_sw128(sKQ + (j & 3) * 2048, 16384, 1024),
                 sdesc_sw128(sXR + j * 2048, 16384, 1024), id2, j > 0);
      if (p.write_O) {
        constexpr uint32_t idp = idesc_tf32(64, R);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mma_tf32(tmem + L::cPU, sdesc_sw128(sP32 + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024),
                   sdesc_sw128(sXR + 16384 + (j >> 2) * (R * 128) + (j & 3) * 32, 16, 1024), idp, j > 0);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    if (!mbar_wait(bar_mma, mma_ph & 1, kWaitNs)) *abort_flag = 1;
    ++mma_ph;
    tc_fence_after();
    // ---------------------------------------------------------------- new state; outputs
    {
      float d2[HALF];
      ld_cols(tmem + lane_base + L::cD2 + half * HALF, d2);
      tmem_ld_wait();
      const float gC = gGam[63];
#pragma unroll
      for (int i = 0; i < HALF; ++i) {
        const int c = half * HALF + i;
        const float s = fmaf(gC, sreg[i], d2[i]);
        sreg[i] = s;
        *reinterpret_cast<float*>(sm + L::S32 + kf32(c, dcol, R)) = tf32r(s);
        const __nv_bfloat16 hi = __float2bfloat16_rn(s);
        *reinterpret_cast<__nv_bfloat16*>(sm + L::SHL + kbf16(c, dcol, R)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sm + L::SHL + R * 256 + kbf16(c, dcol, R)) =
            __float2bfloat16_rn(s - __bfloat162float(hi));
      }
      if (p.write_O) {
        float dq[HALF], pu[HALF];
        ld_cols(tmem + lane_base + L::cD1q + half * HALF, dq);
        ld_cols(tmem + lane_base + L::cPU + half * HALF, pu);
        tmem_ld_wait();
        const int t = 16 * quad + lane;
        if (lane < 16 && t < n) {
          const float gq = gGam[t] * gRq[t];
          __align__(16) __nv_bfloat16 o[HALF];
#pragma unroll
          for (int i = 0; i < HALF; ++i) o[i] = __float2bfloat16_rn(fmaf(gq, dq[i], pu[i]));
          __nv_bfloat16* dst = p.O + ((size_t)(t0 + t) * p.h_v + h) * DV + row0 + half * HALF;
#pragma unroll
          for (int i = 0; i < HALF; i += 8)
            *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<const uint4*>(o + i);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
  }

  if (!ok && tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);
  if (ok) {
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
      const int c = half * HALF + i;
      p.S_out[sbase + (size_t)(row0 + c) * DK + dcol] = sreg[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2D bf16 view [rows][cols] (cols contiguous), 64 x 64 boxes, 128-byte swizzle, zero fill out of range.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R>
cudaError_t launch_scan(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const ScanParams& sp,
                        cudaStream_t stream) {
  using L = ScanLay<R>;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::ALLOC);
  if (e != cudaSuccess) return e;
  chunk_scan_kernel<R><<<dim3(DV / R, sp.h_v, sp.n_seqs), NT, L::ALLOC, stream>>>(mq, mk, mv, sp);
  return cudaGetLastError();
}

}  // namespace

int replay_tc_rows(int n_seqs, int h_v) {
  // few (tail, head) problems: 4 slices of 32 rows per state to fill the SMs; otherwise 2 slices of 64
  return (long long)n_seqs * h_v * 4 <= 2 * 152 ? 32 : 64;
}

bool replay_tc_supported(const SimtParams& p) {
  return p.d_k == DK && p.d_v == DV && p.total_tokens > 0 && p.n_seqs > 0 && !p.augmented;
}

size_t replay_tc_workspace_bytes(int n_seqs, int total_tokens, int h_v) {
  // chunks of all tails <= ceil(total / 64) + one partial chunk per tail
  const size_t chunks = (size_t)(total_tokens + C - 1) / C + (size_t)n_seqs;
  return chunks * (size_t)h_v * kRecBytes;
}

cudaError_t launch_replay_tc(const SimtParams& p, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (workspace_bytes < replay_tc_workspace_bytes(p.n_seqs, p.total_tokens, p.h_v)) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  const void* qsrc = p.write_O ? p.q : p.k;  // q unused without outputs: any valid tile source
  if (!make_map(&mq, qsrc, p.total_tokens, (uint64_t)p.h_k * DK) ||
      !make_map(&mk, p.k, p.total_tokens, (uint64_t)p.h_k * DK) ||
      !make_map(&mv, p.v, p.total_tokens, (uint64_t)p.h_v * DV))
    return cudaErrorInvalidValue;
  unsigned char* rec = static_cast<unsigned char*>(workspace);

  PrepParams pp;
  pp.g = p.g; pp.beta = p.beta; pp.cu = p.cu; pp.rec = rec; pp.status = p.status;
  pp.n_seqs = p.n_seqs; pp.total_tokens = p.total_tokens; pp.h_k = p.h_k; pp.h_v = p.h_v; pp.l2norm = p.l2norm;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PrepLay::ALLOC);
  if (e != cudaSuccess) return e;
  const int chunks_ub = (p.total_tokens + C - 1) / C + p.n_seqs;
  chunk_prep_kernel<<<dim3(chunks_ub, p.h_k), NT, PrepLay::ALLOC, stream>>>(mk, pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ScanParams sp;
  sp.cu = p.cu; sp.S0 = p.S0; sp.rec = rec; sp.O = static_cast<__nv_bfloat16*>(p.O); sp.S_out = p.S_out;
  sp.status = p.status; sp.n_seqs = p.n_seqs; sp.total_tokens = p.total_tokens; sp.h_k = p.h_k; sp.h_v = p.h_v;
  sp.l2norm = p.l2norm; sp.write_O = p.write_O; sp.scale = p.scale;
  return replay_tc_rows(p.n_seqs, p.h_v) == 32 ? launch_scan<32>(mq, mk, mv, sp, stream)
                                               : launch_scan<64>(mq, mk, mv, sp, stream);
}

}  // namespace gdn

// ---------------------------------------------------------------------------------------------
// Allocation-free replay: the same prep + scan kernels, with their scratch in a fixed static
// device array instead of the stream-ordered pool.
// ---------------------------------------------------------------------------------------------
namespace gdn {
namespace {

// 32 MiB on every GPU that loads the library, held until process exit.  Enough for the
// records of one 3277-token tail at 32 v-heads ((52 + 1) chunks x 32 heads x 17408 B).
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, resolved once per device with that device current
// (in host code the symbol itself is only a host-side stand-in).
int static_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(GDN_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= 64) return report_error(GDN_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) return report_error(GDN_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    addr[dev] = ptr;
  }
  *out = addr[dev];
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_replay_noalloc(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
                                  const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out,
                                  float* S_out, void* stream) {
  using namespace gdn;
  SimtParams p;
  bool nothing = false;
  int rc = check_replay_args(dims, q, k, v, g, beta, cu_seqlens, S0, O_out, S_out, &p, &nothing);
  if (rc || nothing) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dims->dtype == GDN_BF16 && !(dims->flags & GDN_PRECISE) && replay_tc_supported(p)) {
    const size_t need = replay_tc_workspace_bytes(p.n_seqs, p.total_tokens, p.h_v);
    if (need > kStaticScratchBytes)
      return report_error(GDN_ERR_NOMEM,
                          "gdn_replay_noalloc: the problem needs more scratch than the 32 MiB static array "
                          "((ceil(total_tokens/64) + n_seqs) * h_v * 17408 bytes); use gdn_replay");
    void* ws = nullptr;
    rc = static_scratch_address(&ws);
    if (rc) return rc;
    const cudaError_t e = launch_replay_tc(p, ws, kStaticScratchBytes, st);
    if (e != cudaSuccess) return report_error(GDN_ERR_CUDA, cudaGetErrorString(e));
    return GDN_OK;
  }
  const cudaError_t e = launch_replay_simt(p, dims->dtype == GDN_BF16, st);  // needs no scratch
  if (e != cudaSuccess) return report_error(GDN_ERR_CUDA, cudaGetErrorString(e));
  return GDN_OK;
}
