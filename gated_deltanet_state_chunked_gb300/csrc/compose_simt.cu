// fp32 CUDA-core composition of chunk operators.
//
// "LinearKV: One Cached State Suffices for Position-Independent Caching in
// Hybrid LLMs", composition passage: chunk j maps an entering state to
// T_{C_j} S + S_local_j (transposed-state form); applying the K maps back to
// back telescopes into the closed form.  In this library's state layout
// (S = d_v x d_k) each step is S <- S T_j^T + S_local_j.  Rows of S evolve
// independently, so one CTA owns a 32-row slice of one head's state and walks
// the K steps, staging T_j in shared memory.
#include "gdn_internal.cuh"
#include "tc_common.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int RS = 32;
constexpr int NT = 256;
constexpr int TST = kMaxHead + 1;  // padded row stride of T in shared memory

__global__ void __launch_bounds__(NT) compose_simt_kernel(ComposeParams p) {
  extern __shared__ __align__(16) float csm[];
  float* Ts = csm;                 // [d_k][TST]
  float* Ss = csm + kMaxHead * TST;  // [RS][TST]
  const int tid = threadIdx.x;
  const int h = blockIdx.y, row0 = blockIdx.x * RS;
  const int DK = p.d_k, DV = p.d_v;
  const size_t sbase = (size_t)h * DV * DK;

  for (int i = tid; i < RS * DK; i += NT) {
    const int r = i / DK, d = i % DK, rg = row0 + r;
    Ss[r * TST + d] = (rg < DV && p.S_in) ? p.S_in[sbase + (size_t)rg * DK + d] : 0.f;
  }
  const int r = tid / 8, c0 = tid % 8;  // thread: row r, columns c0, c0+8, ...
  for (int j = 0; j < p.K; ++j) {
    const float* T = p.T[j] + (size_t)h * DK * DK;
    const float* Sl = p.Slocal[j] + sbase;
    __syncthreads();
    for (int i = tid; i < DK * DK; i += NT) Ts[(i / DK) * TST + (i % DK)] = T[i];
    __syncthreads();
    float acc[kMaxHead / 8];
#pragma unroll
    for (int m = 0; m < kMaxHead / 8; ++m) acc[m] = 0.f;
    for (int kk = 0; kk < DK; ++kk) {
      const float s = Ss[r * TST + kk];
#pragma unroll
      for (int m = 0; m < kMaxHead / 8; ++m) {
        const int i = c0 + 8 * m;
        if (i < DK) acc[m] = fmaf(s, Ts[i * TST + kk], acc[m]);
      }
    }
    const int rg = row0 + r;
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMaxHead / 8; ++m) {
      const int i = c0 + 8 * m;
      if (i < DK) Ss[r * TST + i] = acc[m] + (rg < DV ? Sl[(size_t)rg * DK + i] : 0.f);
    }
  }
  __syncthreads();
  for (int i = tid; i < RS * DK; i += NT) {
    const int rr = i / DK, d = i % DK, rg = row0 + rr;
    if (rg < DV) p.S_out[sbase + (size_t)rg * DK + d] = Ss[rr * TST + d];
  }
}

}  // namespace

cudaError_t launch_compose_simt(const ComposeParams& p, cudaStream_t stream) {
  dim3 grid((p.d_v + RS - 1) / RS, p.h);
  const size_t smem = sizeof(float) * (size_t)(kMaxHead + RS) * TST;
  cudaError_t e = cudaFuncSetAttribute(compose_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  compose_simt_kernel<<<grid, NT, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
