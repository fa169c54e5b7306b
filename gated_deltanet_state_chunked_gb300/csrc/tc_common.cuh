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
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
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

}  // namespace tcp
}  // namespace gdn
