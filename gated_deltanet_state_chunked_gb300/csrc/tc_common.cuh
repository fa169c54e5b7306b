// Shared pieces of the tensor-core path: tile layouts, rounding helpers,
// chunk bookkeeping and the per-(chunk, v-head) record that the prep kernel
// writes and the scan kernel reads.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace tcp {

constexpr int C = kChunk;  // 64 tokens per chunk
constexpr int DK = 128, DV = 128;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on every barrier wait
constexpr float kLog2e = 1.4426950408889634f;

// Record of one (chunk, v-head), written by the prep kernel and copied verbatim into the
// scan kernel's shared memory (the tiles are stored as their 128-byte-swizzled images):
//   [0, 16384)      bf16 [Mb_hi | Mb_lo], Mb = M diag(beta): 2 K-atoms of 64 rows x 128 B
//   [16384, 24576)  bf16 Mw = M diag(beta gamma rk): 1 K-atom of 64 rows x 128 B
//   [24576, 40960)  fp32 P (tf32-rounded), P_ts = rq_t rk_s exp(G_t - G_s) q_t.k_s (s <= t): 2 atoms
//   [40960, 41984)  fp32 gamma_t, rk_t exp(G_last - G_t), gamma_t rq_t, (unused) -- 64 each
// with M = (I + A)^{-1}.  The scan loads [0, 24576) and [24576, 41984) as two parts.
constexpr uint32_t kRecMB = 0, kRecMW = 16384, kRecP = 24576, kRecGate = 40960;
constexpr uint32_t kRecBytes = 41984;
constexpr uint32_t kRecPart1 = 24576, kRecPart2 = kRecBytes - kRecPart1;

__host__ __device__ inline int chunks_of(int len) { return (len + C - 1) / C; }

// Round to the nearest tf32 value (ties away from zero); the tensor cores then read it exactly.
__device__ __forceinline__ float tf32r(float x) {
  // nearest tf32 (10 explicit mantissa bits), ties away from zero, by integer arithmetic on the
  // bit pattern: adding half a tf32 ulp to the magnitude bits carries into the kept bits exactly
  // when the dropped part is at least half an ulp
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

// Upper 16 bits of two floats packed as a bf16 pair (a in the low half): truncation to bf16.
__device__ __forceinline__ uint32_t bf16x2_trunc(float a, float b) {
  return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}
// Two finite floats rounded to the nearest bf16 (ties to even) and packed (a in the low half):
// adding 0x7fff plus the lowest kept bit to the pattern carries into the kept 16 bits exactly
// when the dropped half is above one half ulp, or equal to it with an odd kept part.
__device__ __forceinline__ uint32_t bf16x2_rne(float a, float b) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const uint32_t ra = ua + 0x7fffu + ((ua >> 16) & 1u), rb = ub + 0x7fffu + ((ub >> 16) & 1u);
  return __byte_perm(ra, rb, 0x7632);
}

// Byte offsets inside 128-byte-swizzled tiles (rows of 128 B, 8-row groups of 1024 B).
// fp32 K-major tile, atoms of 32 elements along K, `rows` rows per atom column.
__device__ __forceinline__ uint32_t kf32(uint32_t row, uint32_t k, uint32_t rows) {
  const uint32_t a = k >> 5, c = (k & 31u) * 4u;
  return a * rows * 128u + row * 128u + ((((c >> 4) ^ (row & 7u))) << 4) + (c & 15u);
}
// bf16 K-major tile, atoms of 64 elements along K.
__device__ __forceinline__ uint32_t kbf16(uint32_t row, uint32_t k, uint32_t rows) {
  const uint32_t a = k >> 6, c = (k & 63u) * 2u;
  return a * rows * 128u + row * 128u + ((((c >> 4) ^ (row & 7u))) << 4) + (c & 15u);
}
// bf16 MN-major tile: element (mn, k); atoms of 64 MN-elements, k_rows K-rows per atom.
__device__ __forceinline__ uint32_t mnbf16(uint32_t mn, uint32_t k, uint32_t k_rows) {
  const uint32_t a = mn >> 6, c = (mn & 63u) * 2u;
  return a * k_rows * 128u + k * 128u + ((((c >> 4) ^ (k & 7u))) << 4) + (c & 15u);
}

// Chunk bookkeeping over the packed sequences, block-wide (256 threads).
// Chunks are numbered globally: sequence s owns ceil(len_s / 64) consecutive
// numbers.  Returns the number of chunks before sequence `seq` (*first), the
// total (*total), and, when 0 <= gc < total, the sequence holding global chunk
// gc (*gc_seq) and its index inside it (*gc_idx).  Malformed ranges count as 0
// chunks.  scratch: 16 ints of shared memory.
struct ChunkInfo {
  int first, total, gc_seq, gc_idx;
};

__device__ inline ChunkInfo chunk_info(const int32_t* cu, int n_seqs, int total_tokens, int seq, int gc,
                                       int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n_seqs == 1) {  // one sequence: no scan over the offsets
    const int a = cu[0], b = cu[1];
    const int cnt = (a >= 0 && b >= a && b <= total_tokens) ? chunks_of(b - a) : 0;
    ChunkInfo r;
    r.first = seq == 0 ? 0 : cnt;
    r.total = cnt;
    r.gc_seq = (gc >= 0 && gc < cnt) ? 0 : -1;
    r.gc_idx = (gc >= 0 && gc < cnt) ? gc : 0;
    __syncthreads();
    return r;
  }
  if (tid == 0) { scratch[8] = 0; scratch[9] = -1; scratch[10] = 0; }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < n_seqs; base += 256) {
    const int i = base + tid;
    int cnt = 0;
    if (i < n_seqs) {
      const int a = cu[i], b = cu[i + 1];
      cnt = (a >= 0 && b >= a && b <= total_tokens) ? chunks_of(b - a) : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int wsum = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int s = scratch[w];
      if (w < warp) wsum += s;
      all += s;
    }
    const int excl = carry + wsum + incl - cnt;
    if (i < n_seqs && i == seq) scratch[8] = excl;
    if (i < n_seqs && cnt > 0 && gc >= excl && gc < excl + cnt) { scratch[9] = i; scratch[10] = gc - excl; }
    carry += all;
    __syncthreads();
  }
  ChunkInfo r;
  r.first = (seq >= 0 && seq < n_seqs) ? scratch[8] : carry;
  r.total = carry;
  r.gc_seq = scratch[9];
  r.gc_idx = scratch[10];
  __syncthreads();
  return r;
}

// Named barrier over one 128-thread warpgroup (ids 1, 2, ...; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

constexpr int MST = 68;  // row stride (floats) of the 64x64 fp32 work matrices (16-byte aligned rows)

// M = (I + A)^{-1} for a 64x64 strictly lower A (stride MST), by one 128-thread warpgroup
// (t = thread index in the group, bid = its named barrier).  In 32x32 blocks,
//   M11 = (I + A11)^{-1}, M22 = (I + A22)^{-1}, M21 = -M22 A21 M11, M12 = 0:
// the diagonal blocks by forward substitution with one column per thread held in registers
// (each row of A is a broadcast load), then the two products with 8 outputs per thread.  A's
// upper-right block (zero, unused afterwards) holds A21 M11 in between.
__device__ inline void invert_unit_lower(float* A, float* M, int t, int bid) {
  if (t < 64) {
    const int b = t >> 5, j = t & 31;
    const float* Ab = A + (32 * b) * MST + 32 * b;
    float m[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int s = 0; s + 3 < r; s += 4) {
        const float4 a = *reinterpret_cast<const float4*>(Ab + r * MST + s);
        a0 = fmaf(a.x, m[s], a0);
        a1 = fmaf(a.y, m[s + 1], a1);
        a2 = fmaf(a.z, m[s + 2], a2);
        a3 = fmaf(a.w, m[s + 3], a3);
      }
#pragma unroll
      for (int s = r & ~3; s < r; ++s) a0 = fmaf(Ab[r * MST + s], m[s], a0);
      const float x = -((a0 + a1) + (a2 + a3));
      m[r] = r == j ? 1.f : (r < j ? 0.f : x);
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) M[(32 * b + r) * MST + 32 * b + j] = m[r];
  } else {
    for (int i = t - 64; i < 256; i += 64)  // M12 = 0
      *reinterpret_cast<float4*>(M + (i >> 3) * MST + 32 + (i & 7) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  group_sync(bid);
  const int r = t >> 2, c8 = (t & 3) * 8;  // output rows r of a 32x32 block, columns [c8, c8 + 8)
  {  // X = A21 M11 -> A[0:32][32:64]
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.f;
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float a = A[(32 + r) * MST + k];
      const float4 m0 = *reinterpret_cast<const float4*>(M + k * MST + c8);
      const float4 m1 = *reinterpret_cast<const float4*>(M + k * MST + c8 + 4);
      x[0] = fmaf(a, m0.x, x[0]); x[1] = fmaf(a, m0.y, x[1]); x[2] = fmaf(a, m0.z, x[2]); x[3] = fmaf(a, m0.w, x[3]);
      x[4] = fmaf(a, m1.x, x[4]); x[5] = fmaf(a, m1.y, x[5]); x[6] = fmaf(a, m1.z, x[6]); x[7] = fmaf(a, m1.w, x[7]);
    }
    *reinterpret_cast<float4*>(A + r * MST + 32 + c8) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(A + r * MST + 32 + c8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
  group_sync(bid);
  {  // M21 = -M22 X
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = 0.f;
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float mm = M[(32 + r) * MST + 32 + k];
      const float4 x0 = *reinterpret_cast<const float4*>(A + k * MST + 32 + c8);
      const float4 x1 = *reinterpret_cast<const float4*>(A + k * MST + 32 + c8 + 4);
      y[0] = fmaf(mm, x0.x, y[0]); y[1] = fmaf(mm, x0.y, y[1]); y[2] = fmaf(mm, x0.z, y[2]); y[3] = fmaf(mm, x0.w, y[3]);
      y[4] = fmaf(mm, x1.x, y[4]); y[5] = fmaf(mm, x1.y, y[5]); y[6] = fmaf(mm, x1.z, y[6]); y[7] = fmaf(mm, x1.w, y[7]);
    }
    *reinterpret_cast<float4*>(M + (32 + r) * MST + c8) = make_float4(-y[0], -y[1], -y[2], -y[3]);
    *reinterpret_cast<float4*>(M + (32 + r) * MST + c8 + 4) = make_float4(-y[4], -y[5], -y[6], -y[7]);
  }
  group_sync(bid);
}

}  // namespace tcp
}  // namespace gdn
