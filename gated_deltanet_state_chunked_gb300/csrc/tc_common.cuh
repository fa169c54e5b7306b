// Shared pieces of the tensor-core path: tile layouts, rounding helpers,
// chunk bookkeeping and the per-(chunk, v-head) record that the prep kernel
// writes and the scan kernel reads.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include <climits>

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

// Chunk bookkeeping over the packed sequences, block-wide (NW warps, the whole CTA).
// Chunks are numbered globally: sequence s owns ceil(len_s / 64) consecutive
// numbers.  A range [cu[i], cu[i+1]) counts only when 0 <= cu[i] <= cu[i+1] <=
// total_tokens and cu[i] is at least every earlier offset (the offsets are
// non-decreasing up to i); the counted ranges are then disjoint, so they hold
// at most ceil(total_tokens / 64) + n_seqs chunks, the size of every per-chunk
// buffer.  Other ranges count as 0 chunks and are not valid.  Returns the number
// of chunks before sequence `seq` (*first), whether `seq` is valid, the total,
// and, when 0 <= gc < total, the sequence holding global chunk gc (*gc_seq) and
// its index inside it (*gc_idx).  scratch: 2 NW + 4 ints of shared memory.
struct ChunkInfo {
  int first, total, gc_seq, gc_idx;
  bool valid;
};

template <int NW>
__device__ inline ChunkInfo chunk_info_n(const int32_t* cu, int n_seqs, int total_tokens, int seq, int gc,
                                         int* scratch) {
  constexpr int NTH = 32 * NW;  // offsets examined per round
  constexpr int RS = 2 * NW;    // results: first, gc_seq, gc_idx, valid
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n_seqs == 1) {  // one sequence: no scan over the offsets
    const int a = cu[0], b = cu[1];
    const bool ok = a >= 0 && b >= a && b <= total_tokens;
    const int cnt = ok ? chunks_of(b - a) : 0;
    ChunkInfo r;
    r.first = seq == 0 ? 0 : cnt;
    r.total = cnt;
    r.valid = seq == 0 && ok;
    r.gc_seq = (gc >= 0 && gc < cnt) ? 0 : -1;
    r.gc_idx = (gc >= 0 && gc < cnt) ? gc : 0;
    __syncthreads();
    return r;
  }
  if (tid == 0) { scratch[RS] = 0; scratch[RS + 1] = -1; scratch[RS + 2] = 0; scratch[RS + 3] = 0; }
  __syncthreads();
  int carry = 0;                // chunks of the ranges before this round's block of offsets
  int carry_max = cu[0];        // largest offset before this round's ranges
  for (int base = 0; base < n_seqs; base += NTH) {
    const int i = base + tid;
    int a = 0, b = INT_MIN;
    if (i < n_seqs) { a = cu[i]; b = cu[i + 1]; }
    // largest end offset of the ranges before i: exclusive prefix maximum of b
    int incl = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl = max(incl, x);
    }
    int excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = INT_MIN;
    if (lane == 31) scratch[NW + warp] = incl;
    __syncthreads();
    int wmax = INT_MIN, allmax = INT_MIN;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int m = scratch[NW + w];
      if (w < warp) wmax = max(wmax, m);
      allmax = max(allmax, m);
    }
    const int before = max(carry_max, max(wmax, excl));
    const bool ok = i < n_seqs && a >= 0 && a >= before && b >= a && b <= total_tokens;
    const int cnt = ok ? chunks_of(b - a) : 0;
    int inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    int wsum = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int s = scratch[w];
      if (w < warp) wsum += s;
      all += s;
    }
    const int ex = carry + wsum + inc - cnt;
    if (i < n_seqs && i == seq) { scratch[RS] = ex; scratch[RS + 3] = ok ? 1 : 0; }
    if (cnt > 0 && gc >= ex && gc < ex + cnt) { scratch[RS + 1] = i; scratch[RS + 2] = gc - ex; }
    carry += all;
    carry_max = max(carry_max, allmax);
    __syncthreads();
  }
  ChunkInfo r;
  r.first = (seq >= 0 && seq < n_seqs) ? scratch[RS] : carry;
  r.valid = (seq >= 0 && seq < n_seqs) && scratch[RS + 3] != 0;
  r.total = carry;
  r.gc_seq = scratch[RS + 1];
  r.gc_idx = scratch[RS + 2];
  __syncthreads();
  return r;
}
// The 256-thread kernels' form (scratch: 20 ints).
__device__ inline ChunkInfo chunk_info(const int32_t* cu, int n_seqs, int total_tokens, int seq, int gc,
                                       int* scratch) {
  return chunk_info_n<8>(cu, n_seqs, total_tokens, seq, gc, scratch);
}

// Named barrier over one 128-thread warpgroup (ids 1, 2, ...; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
// Producer / consumer hand-off on named barrier `id` with `count` participating threads in all
// (a multiple of 32): producers arrive without waiting, consumers wait until every participant
// has reached it.  Memory operations before the arrival are visible to the consumers after it.
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

constexpr int MST = 68;  // row stride (floats) of the 64x64 fp32 work matrices (16-byte aligned rows)

// One warp-level tensor-core product D(16x8) += A(16x8) B(8x8), tf32 inputs, fp32 accumulate
// (the legacy mma.sync path: enough for 32x32 blocks that are too small for tcgen05).
// Fragments: A rows g and g+8, columns q and q+4; B rows q and q+4, column g; D rows g and
// g+8, columns 2q and 2q+1 (g = lane / 4, q = lane % 4).
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// x = hi + lo with hi = x truncated to tf32 (low 13 mantissa bits cleared); lo is exact in fp32
// and is itself read as tf32 by the product, so hi*hi' + hi*lo' + lo*hi' carries about 21
// significant bits.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

// As split_tf32 with hi the nearest tf32 value of x (ties away from zero): |lo| <= 2^-11 |x|.
__device__ __forceinline__ void split_tf32_rn(float x, uint32_t& hi, uint32_t& lo) {
  const float h = tf32r(x);
  hi = __float_as_uint(h);
  lo = __float_as_uint(x - h);
}

// One warp: acc[j] (the 16 x 8 tile at rows [m0, m0 + 16), columns [n0 + 8 j, +8)) += the sum
// over k in [k_lo, k_hi) (multiples of 8) of a(m, k) b(k, n), on the warp-level tensor cores in
// split tf32 (hi = nearest tf32, lo = the rest; lo*hi' + hi*lo' + hi*hi', about 21 bits).
// Tiles with n0 + 8 j >= n_lim are skipped.  a and b read shared memory; the fragments follow
// the m16n8k8 layout (see mma_m16n8k8_tf32).
template <int NTL, typename FA, typename FB>
__device__ __forceinline__ void warp_mma_tf32x3(float (&acc)[NTL][4], FA a, FB b, int m0, int n0, int k_lo,
                                                int k_hi, int n_lim) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll 4
  for (int k0 = k_lo; k0 < k_hi; k0 += 8) {
    uint32_t ah[4], al[4];
    split_tf32_rn(a(m0 + g, k0 + q), ah[0], al[0]);
    split_tf32_rn(a(m0 + g + 8, k0 + q), ah[1], al[1]);
    split_tf32_rn(a(m0 + g, k0 + q + 4), ah[2], al[2]);
    split_tf32_rn(a(m0 + g + 8, k0 + q + 4), ah[3], al[3]);
#pragma unroll
    for (int j = 0; j < NTL; ++j) {
      const int n = n0 + 8 * j;
      if (n >= n_lim) continue;
      uint32_t bh[2], bl[2];
      split_tf32_rn(b(k0 + q, n + g), bh[0], bl[0]);
      split_tf32_rn(b(k0 + q + 4, n + g), bh[1], bl[1]);
      mma_m16n8k8_tf32(acc[j], al, bh);
      mma_m16n8k8_tf32(acc[j], ah, bl);
      mma_m16n8k8_tf32(acc[j], ah, bh);
    }
  }
}

// D = sign * L R for 32x32 blocks of stride MST, by one 128-thread warpgroup (t = thread index
// in it): warp w computes rows [16 (w / 2), +16) and columns [16 (w % 2), +16) with three
// tf32 products per 8x8 step (split operands).
__device__ inline void block_mm32(const float* L, const float* Rm, float* D, float sign, int t) {
  const int w = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  const int r0 = 16 * (w >> 1), c0 = 16 * (w & 1);
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int k0 = 0; k0 < 32; k0 += 8) {
    uint32_t ah[4], al[4];
    split_tf32(L[(r0 + g) * MST + k0 + q], ah[0], al[0]);
    split_tf32(L[(r0 + g + 8) * MST + k0 + q], ah[1], al[1]);
    split_tf32(L[(r0 + g) * MST + k0 + q + 4], ah[2], al[2]);
    split_tf32(L[(r0 + g + 8) * MST + k0 + q + 4], ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n = c0 + 8 * nt + g;
      uint32_t bh[2], bl[2];
      split_tf32(Rm[(k0 + q) * MST + n], bh[0], bl[0]);
      split_tf32(Rm[(k0 + q + 4) * MST + n], bh[1], bl[1]);
      mma_m16n8k8_tf32(acc[nt], al, bh);
      mma_m16n8k8_tf32(acc[nt], ah, bl);
      mma_m16n8k8_tf32(acc[nt], ah, bh);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int c = c0 + 8 * nt + 2 * q;
    *reinterpret_cast<float2*>(D + (r0 + g) * MST + c) = make_float2(sign * acc[nt][0], sign * acc[nt][1]);
    *reinterpret_cast<float2*>(D + (r0 + g + 8) * MST + c) = make_float2(sign * acc[nt][2], sign * acc[nt][3]);
  }
}

// D = sign * L R for 16x16 blocks of stride MST, by one warp (three tf32 products per 8x8 step,
// split operands as in block_mm32).
__device__ inline void block_mm16(const float* L, const float* Rm, float* D, float sign) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int k0 = 0; k0 < 16; k0 += 8) {
    uint32_t ah[4], al[4];
    split_tf32(L[g * MST + k0 + q], ah[0], al[0]);
    split_tf32(L[(g + 8) * MST + k0 + q], ah[1], al[1]);
    split_tf32(L[g * MST + k0 + q + 4], ah[2], al[2]);
    split_tf32(L[(g + 8) * MST + k0 + q + 4], ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n = 8 * nt + g;
      uint32_t bh[2], bl[2];
      split_tf32(Rm[(k0 + q) * MST + n], bh[0], bl[0]);
      split_tf32(Rm[(k0 + q + 4) * MST + n], bh[1], bl[1]);
      mma_m16n8k8_tf32(acc[nt], al, bh);
      mma_m16n8k8_tf32(acc[nt], ah, bl);
      mma_m16n8k8_tf32(acc[nt], ah, bh);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int c = 8 * nt + 2 * q;
    *reinterpret_cast<float2*>(D + g * MST + c) = make_float2(sign * acc[nt][0], sign * acc[nt][1]);
    *reinterpret_cast<float2*>(D + (g + 8) * MST + c) = make_float2(sign * acc[nt][2], sign * acc[nt][3]);
  }
}

// M = (I + A)^{-1} for a 64x64 strictly lower A (stride MST), by one 128-thread warpgroup
// (t = thread index in the group, bid = its named barrier).  For a unit lower block matrix
// [[I + X, 0], [Y, I + Z]] the inverse is [[P, 0], [-Q Y P, Q]] with P = (I + X)^{-1},
// Q = (I + Z)^{-1}; applied twice:
//  * warps 0 and 1 solve the four 16x16 diagonal blocks by forward substitution, one column
//    per thread held in registers (each row of A is a broadcast load), and each merges its
//    pair into a 32x32 diagonal block, while the other two warps clear the upper blocks of M;
//  * the warpgroup merges those two into M.
// The products run on the warp-level tensor cores in split tf32 (about fp32 accuracy).  A's
// upper blocks (zero, unused afterwards) hold the intermediate Y P products.
__device__ inline void invert_unit_lower(float* A, float* M, int t, int bid) {
  if (t < 64) {
    const int b = t >> 4, j = t & 15;
    const float* Ab = A + (16 * b) * MST + 16 * b;
    float m[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
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
    for (int r = 0; r < 16; ++r) M[(16 * b + r) * MST + 16 * b + j] = m[r];
    // warp w: 32x32 diagonal block w from its two 16x16 blocks (both solved by this warp)
    __syncwarp();
    const int o = 32 * (t >> 5);
    block_mm16(A + (o + 16) * MST + o, M + o * MST + o, A + o * MST + o + 16, 1.f);  // Y P
    __syncwarp();
    block_mm16(M + (o + 16) * MST + o + 16, A + o * MST + o + 16, M + (o + 16) * MST + o, -1.f);  // -Q (Y P)
  } else {
    // upper blocks of M: rows 0-31 x columns 32-63, rows 0-15 x 16-31, rows 32-47 x 48-63
    for (int i = t - 64; i < 384; i += 64) {
      int row, col;
      if (i < 256) {
        row = i >> 3, col = 32 + (i & 7) * 4;
      } else if (i < 320) {
        row = (i - 256) >> 2, col = 16 + (i & 3) * 4;
      } else {
        row = 32 + ((i - 320) >> 2), col = 48 + (i & 3) * 4;
      }
      *reinterpret_cast<float4*>(M + row * MST + col) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  group_sync(bid);
  block_mm32(A + 32 * MST, M, A + 32, 1.f, t);                   // A21 M11 -> A[0:32][32:64]
  group_sync(bid);
  block_mm32(M + 32 * MST + 32, A + 32, M + 32 * MST, -1.f, t);  // M21 = -M22 (A21 M11)
  group_sync(bid);
}

}  // namespace tcp
}  // namespace gdn
