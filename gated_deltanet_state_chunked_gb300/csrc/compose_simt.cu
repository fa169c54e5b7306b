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

// ---------------------------------------------------------------------------------------------
// d_k = d_v = 128: register-tiled kernel.  One CTA owns 32 rows of one head's state (kept in
// shared memory) and walks the K steps.  T_j (64 KB, contiguous) and S_local_j's 32-row slice
// arrive by bulk copies two steps ahead of use.  Thread (b, g) of each 128-thread half computes
// rows 4 b .. 4 b + 3 and columns g + 16 i (i < 8) of S T_j^T over its half of k with float4
// shared loads (each loaded T value feeds four rows, each S value eight columns), walking k in an
// order rotated by 4 g so that the eight threads of a quarter warp read eight different 16-byte
// chunks of their T and S rows; the second half's partial sums are added through shared memory.
constexpr int CR = 32, CNT = 256, CPAD = 132, CD = 128;
struct CLay {
  static constexpr uint32_t TB = 0;                       // 2 x T_j [128][128] fp32
  static constexpr uint32_t TBYTES = CD * CD * 4;         // 65536
  static constexpr uint32_t SS = 2 * TBYTES;              // S slice [32][132]
  static constexpr uint32_t LB = SS + CR * CPAD * 4;      // 2 x S_local slice [32][128]
  static constexpr uint32_t RED = LB + 2 * CR * CD * 4;   // partial sums of the second k half [32][128]
  static constexpr uint32_t BARS = RED + CR * CD * 4;     // bar_t[2], bar_l[2], abort flag
  static constexpr uint32_t TOTAL = BARS + 64;
};

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(CNT, 1) compose_tiled_kernel(ComposeParams p) {
  using L = CLay;
  extern __shared__ __align__(16) unsigned char cmem[];
  float* Sx = reinterpret_cast<float*>(cmem + L::SS);
  uint64_t* bar_t = reinterpret_cast<uint64_t*>(cmem + L::BARS);
  uint64_t* bar_l = bar_t + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cmem + L::BARS + 32);
  const int tid = threadIdx.x, lane = tid & 31, kh = tid >> 7, rb = 4 * ((tid & 127) >> 4), g = tid & 15;
  float* Red = reinterpret_cast<float*>(cmem + L::RED);
  const int h = blockIdx.y, row0 = blockIdx.x * CR;
  const size_t sbase = (size_t)h * CD * CD;

  auto issue_t = [&](int j) {  // warp 0
    unsigned char* dst = cmem + L::TB + (j & 1) * L::TBYTES;
    if (lane == 0) {
      tc::mbar_arrive_expect_tx(&bar_t[j & 1], CD * CD * 4);
      const float* src = p.T[j] + sbase;
      bulk_copy(dst, src, CD * CD * 2, &bar_t[j & 1]);
      bulk_copy(dst + CD * CD * 2, src + CD * CD / 2, CD * CD * 2, &bar_t[j & 1]);
    }
  };
  auto issue_l = [&](int j) {  // one thread
    tc::mbar_arrive_expect_tx(&bar_l[j & 1], CR * CD * 4);
    bulk_copy(cmem + L::LB + (j & 1) * (CR * CD * 4), p.Slocal[j] + sbase + (size_t)row0 * CD, CR * CD * 4,
              &bar_l[j & 1]);
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (*abort_flag) return;
    if (!tc::mbar_wait(bar, parity, tcp::kWaitNs)) *abort_flag = 1;
  };

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::mbar_init(&bar_t[i], 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
  }
  for (int i = tid; i < CR * CD; i += CNT) {
    const int rr = i / CD, d = i % CD;
    Sx[rr * CPAD + d] = p.S_in ? p.S_in[sbase + (size_t)(row0 + rr) * CD + d] : 0.f;
  }
  __syncthreads();
  if (tid < 32) {
    for (int j = 0; j < 2 && j < p.K; ++j) {
      issue_t(j);
      if (lane == 0) issue_l(j);
    }
  }
  for (int j = 0; j < p.K; ++j) {
    const uint32_t par = (j >> 1) & 1;
    const float* Tb = reinterpret_cast<const float*>(cmem + L::TB + (j & 1) * L::TBYTES);
    wait(&bar_t[j & 1], par);
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[a][i] = 0.f;
#pragma unroll 2
    for (int q = 0; q < CD / 8; ++q) {
      const int kk = (kh * (CD / 8) + ((q + g) & (CD / 8 - 1))) * 4;
      float4 s4[4], t4[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) s4[a] = *reinterpret_cast<const float4*>(Sx + (rb + a) * CPAD + kk);
#pragma unroll
      for (int i = 0; i < 8; ++i) t4[i] = *reinterpret_cast<const float4*>(Tb + (g + 16 * i) * CD + kk);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[a][i] = fmaf(s4[a].x, t4[i].x, acc[a][i]);
          acc[a][i] = fmaf(s4[a].y, t4[i].y, acc[a][i]);
          acc[a][i] = fmaf(s4[a].z, t4[i].z, acc[a][i]);
          acc[a][i] = fmaf(s4[a].w, t4[i].w, acc[a][i]);
        }
    }
    if (kh == 1) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int i = 0; i < 8; ++i) Red[(rb + a) * CD + g + 16 * i] = acc[a][i];
    }
    __syncthreads();  // every read of the state slice and of T_j is done; partial sums are in place
    if (tid < 32 && j + 2 < p.K) issue_t(j + 2);
    wait(&bar_l[j & 1], par);
    const float* Lb = reinterpret_cast<const float*>(cmem + L::LB + (j & 1) * (CR * CD * 4));
    if (kh == 0) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int o = (rb + a) * CD + g + 16 * i;
          Sx[(rb + a) * CPAD + g + 16 * i] = (acc[a][i] + Red[o]) + Lb[o];
        }
    }
    __syncthreads();  // the new state slice is complete; S_local_j's buffer is free
    if (tid == 0 && j + 2 < p.K) issue_l(j + 2);
  }
  if (*abort_flag) {
    if (tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);
    return;
  }
  for (int i = tid; i < CR * CD; i += CNT) {
    const int rr = i / CD, d = i % CD;
    p.S_out[sbase + (size_t)(row0 + rr) * CD + d] = Sx[rr * CPAD + d];
  }
}

}  // namespace

cudaError_t launch_compose_simt(const ComposeParams& p, cudaStream_t stream) {
  if (p.d_k == CD && p.d_v == CD) {
    cudaError_t e = cudaFuncSetAttribute(compose_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)CLay::TOTAL);
    if (e != cudaSuccess) return e;
    compose_tiled_kernel<<<dim3(CD / CR, p.h), CNT, CLay::TOTAL, stream>>>(p);
    return cudaGetLastError();
  }
  dim3 grid((p.d_v + RS - 1) / RS, p.h);
  const size_t smem = sizeof(float) * (size_t)(kMaxHead + RS) * TST;
  cudaError_t e = cudaFuncSetAttribute(compose_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  compose_simt_kernel<<<grid, NT, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
