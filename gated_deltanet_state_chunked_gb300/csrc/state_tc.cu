// Operator-form chunked scan for state-only replay (bf16 inputs, d_k = d_v = 128, 32-row slices).
//
// Method: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix Caching for Hybrid
// LLMs", section 2 Eq. (1) and section 3 Eq. (2), chunk by chunk (C = 64 tokens), with the same
// per-chunk quantities as the tensor-core scan (replay_tc.cu): M = (I + A)^{-1},
// U~ = M diag(beta) V, W = M diag(beta gamma rk) K, sc_t = rk_t exp(G_C - G_t).  The state step
//   S^T <- gamma_C S^T + K^T diag(sc) (U~ - W S^T)
// is regrouped around the chunk's d_k x d_k operator so that the chunk-to-chunk chain holds a
// single contraction:
//   S^T <- gamma_C S^T + B^T + A^T S^T,    A^T = K^T Z K,   B^T = K^T diag(sc) U~,
// with Z = -diag(sc) Mw (Mw = M diag(beta gamma rk), stored by the prep kernel in place of Mw
// when this scan follows).  A^T and B^T do not depend on the state: they are built one to two
// chunks ahead of the chain.  (W S^T is never formed; outputs are not produced here.)
//
// Per chunk, per CTA (one 32-row slice of one (tail, v-head) state), all accumulated in fp32 in
// TMEM (lane = row of the M=128 layout):
//   U~  = [Mb_hi | Mb_lo] [V; V]        bf16 (Mb split hi + lo)          M=128 N=32  K=128
//   Y   = K^T Z                         bf16 (Z rounded once)            M=128 N=64  K=64
//   A^T = [Y_hi | Y_lo] [K; K]          bf16 (Y split hi + lo)           M=128 N=128 K=128
//   B^T = K^T [U~s_hi | U~s_lo]         bf16 (U~s = diag(sc) U~ split)    M=128 N=64  K=64
//   D  += A^T S^T                       tf32, A^T from TMEM, two warps   M=128 N=32  K=128
//                                       (K halves into the [hi | lo] halves of B^T)
//   S  <- gamma_C S + D_hi + D_lo       fp32 registers; S^T written back tf32-rounded
//
// Warp roles (13 warps): 0-3 the chain (warps 0-1 issue the chain product, all four update the
// state), 4-7 epilogues (Y split by 4-7, U~s by 4-5: the TMEM lane quarters of each warp), 8 the
// loads, 9-12 one MMA group each (U~, Y, A^T, B^T).  Hand-offs are mbarriers, one per buffer
// slot and chunk residue, placed so that the next completion of the barrier a role polls always
// depends on something that role does after the poll (a parity wait then never sees two phases
// complete at once); each wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace tcp;

constexpr int SR = 32;             // state rows per CTA
constexpr int SW = 13;             // warps
constexpr int SNT = SW * 32;
constexpr int NKB = 3;             // K tile buffers
constexpr uint32_t kFac = 512;     // per-chunk factors: gamma_t, rk_t exp(G_last - G_t)
constexpr uint64_t kDrainNs = 10000000ull;  // bound on the final waits for copies and products

struct StLay {
  static constexpr uint32_t KB = 0;                    // NKB x bf16 K tile: 2 d_k atoms x (64 rows x 128 B)
  static constexpr uint32_t VB = KB + NKB * 16384;     // 2 x bf16 V atom: 64 tokens x 128 B
  static constexpr uint32_t R1 = VB + 2 * 8192;        // 2 x record part 1: [Mb_hi | Mb_lo] (16 KB), Z (8 KB)
  static constexpr uint32_t YS = R1 + 2 * kRecPart1;   // 2 x bf16 [Y_hi | Y_lo]: 2 K atoms x (128 rows x 128 B)
  static constexpr uint32_t UH = YS + 2 * 32768;       // 2 x bf16 [U~s_hi | U~s_lo], MN-major, 64 tokens x 128 B
  static constexpr uint32_t S32 = UH + 2 * 8192;       // fp32 state slice (32 rows x 4 atoms), tf32-rounded
  static constexpr uint32_t FB = S32 + SR * 512;       // 4 x factors
  static constexpr uint32_t BARS = FB + 4 * kFac;
  static constexpr uint32_t TOTAL = BARS + 512;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM columns
  static constexpr uint32_t cA = 0;    // 2 x 128: A^T (fp32), the chain product's A operand
  static constexpr uint32_t cY = 256;  // 64: Y
  static constexpr uint32_t cC = 320;  // 2 x 64: [hi | lo] = B^T halves, then + the chain halves
  static constexpr uint32_t cU = 448;  // 2 x 32: U~
  static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(StLay::ALLOC <= 232448, "shared memory");
static_assert(StLay::R1 % 1024 == 0 && StLay::YS % 1024 == 0 && StLay::UH % 1024 == 0 && StLay::S32 % 1024 == 0 &&
                  kRecPart1 % 1024 == 0 && kRecMW % 1024 == 0,
              "tile alignment");

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Advance a shared-memory descriptor's start address by a byte offset (multiple of 16).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

template <int J0, int J1, typename F>
__device__ __forceinline__ void issue_range(F&& f) {
#pragma unroll
  for (int j = J0; j < J1; ++j) f(j, j == J0);
}

// bf16 truncation of x as a float
__device__ __forceinline__ float hi16(float x) { return __uint_as_float(__float_as_uint(x) & 0xffff0000u); }

__global__ void __launch_bounds__(SNT, 1)
    chunk_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                       StateParams p) {
  using L = StLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_k = bars + 0;    // [3] K tile of chunk c (slot c % 3)
  uint64_t* bar_vr = bars + 3;   // [2] V atom and record part 1 of chunk c (slot c & 1)
  uint64_t* bar_f = bars + 5;    // [4] factors of chunk c (slot c & 3)
  uint64_t* bar_u = bars + 9;    // [2] U~(c) in cU slot c & 1
  uint64_t* bar_y = bars + 11;   // [2] Y(c) in cY (slot c & 1)
  uint64_t* bar_ys = bars + 13;  // [4] Y(c) read out of cY and split into YS slot c & 1 (4 warps)
  uint64_t* bar_uh = bars + 17;  // [4] U~(c) read out of cU, U~s(c) in UH slot c & 1 (2 warps)
  uint64_t* bar_a = bars + 21;   // [4] A^T(c) in cA slot c & 1
  uint64_t* bar_b = bars + 25;   // [4] B^T(c) in cC slot c & 1
  uint64_t* bar_c = bars + 29;   // [4] chain product of chunk c (2 issuing warps)
  uint64_t* bar_s = bars + 33;   // [4] state update of chunk c done: cC slot c & 1 read
  uint64_t* bar_dr = bars + 37;  // final commit of every issuing warp (6)
  constexpr int NBARS = 38;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 304);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + L::BARS + 308);
  int* scratch = reinterpret_cast<int*>(sm + L::BARS + 320);  // chunk_info_n<13>: 30 ints

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const int slice = blockIdx.x, h = blockIdx.y, seq = p.order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int row0 = slice * SR;
  const int hk = h / (p.h_v / p.h_k);

  // A malformed range (see chunk_info) has no records: report it before forming any address.
  const ChunkInfo ci = chunk_info_n<SW>(p.cu, p.n_seqs, p.total_tokens, seq, -1, scratch);
  if (!ci.valid) {
    if (tid == 0) atomicExch(p.status, GDN_ERR_SHAPE);
    return;
  }
  const int t_begin = p.cu[seq], t_end = p.cu[seq + 1];
  const int nch = chunks_of(t_end - t_begin);

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  auto rec_of = [&](int c) { return p.rec + ((size_t)(ci.first + c) * p.h_v + h) * kRecBytes; };
  auto load_k = [&](int c) {  // one thread
    uint64_t* b = &bar_k[c % NKB];
    mbar_arrive_expect_tx(b, 16384);
    for (int a = 0; a < 2; ++a)
      tma_load_2d(sm + L::KB + (c % NKB) * 16384 + a * 8192, &map_k, b, hk * DK + a * 64, t_begin + c * C);
  };
  auto load_vr = [&](int c) {  // one thread
    uint64_t* b = &bar_vr[c & 1];
    mbar_arrive_expect_tx(b, 8192 + kRecPart1);
    tma_load_2d(sm + L::VB + (c & 1) * 8192, &map_v, b, h * DV + (row0 & ~63), t_begin + c * C);
    bulk_g2s(sm + L::R1 + (c & 1) * kRecPart1, rec_of(c), kRecPart1, b);
  };
  auto load_f = [&](int c) {  // one thread
    uint64_t* b = &bar_f[c & 3];
    mbar_arrive_expect_tx(b, kFac);
    bulk_g2s(sm + L::FB + (c & 3) * kFac, rec_of(c) + kRecGate, kFac, b);
  };
  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {
      const uint64_t* b = &bars[i];
      const int n = (b >= bar_ys && b < bar_ys + 4) ? 4 : (b >= bar_uh && b < bar_uh + 4) ? 2
                    : (b >= bar_c && b < bar_c + 4) ? 2 : b == bar_dr ? 6 : 1;
      mbar_init(&bars[i], n);
    }
    mbar_fence_init();
    flags[0] = 0;
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    for (int c = 0; c < min(nch, NKB); ++c) load_k(c);  // inputs: no wait for the prep kernel
    grid_dep_wait();                                     // the records are written by the prep kernel
    for (int c = 0; c < min(nch, 2); ++c) load_vr(c);
    for (int c = 0; c < min(nch, 4); ++c) load_f(c);
  }
  grid_dep_wait();

  // entering state (chain warps): thread owns d_k column 32*quad + lane and all 32 rows
  const int dcol = 32 * quad + lane;
  float sreg[SR];
  const size_t sbase = ((size_t)seq * p.h_v + h) * DV * DK;
  if (warp < 4) {
#pragma unroll
    for (int r = 0; r < SR; ++r) {
      const float s = p.S0 ? p.S0[sbase + (size_t)(row0 + r) * DK + dcol] : 0.f;
      sreg[r] = s;
      *reinterpret_cast<float*>(sm + L::S32 + kf32(r, dcol, SR)) = tf32r(s);
    }
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t vcoloff = (uint32_t)(row0 & 63) * 2u;
  const uint64_t dK = sdesc_sw128(smem_u32(sm + L::KB), 8192, 1024);          // MN-major K (as K^T or as K)
  const uint64_t dV = sdesc_sw128(smem_u32(sm + L::VB) + vcoloff, 8192, 1024);  // MN-major V slice
  const uint64_t dMb = sdesc_sw128(smem_u32(sm + L::R1), 16, 1024);            // K-major [Mb_hi | Mb_lo]
  const uint64_t dZ = sdesc_sw128(smem_u32(sm + L::R1 + kRecMW), 8192, 1024);  // MN-major Z
  const uint64_t dYS = sdesc_sw128(smem_u32(sm + L::YS), 16, 1024);            // K-major [Y_hi | Y_lo]
  const uint64_t dUH = sdesc_sw128(smem_u32(sm + L::UH), 8192, 1024);          // MN-major [U~s_hi | U~s_lo]
  const uint64_t dS32 = sdesc_sw128(smem_u32(sm + L::S32), 16, 1024);          // K-major S (tf32)
  // Bounded wait, suspending rather than spinning (a polling warp takes issue slots from the
  // warps that share its scheduler: the epilogues sit beside the chain warps).  After the first
  // timeout every later wait returns at once and no further copy or product is issued, so every
  // role runs its loop to the end and the CTA reports the error.
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (flags[0]) return;
    if (!mbar_wait(bar, parity, kWaitNs)) flags[0] = 1;
  };
  auto live = [&]() { return flags[0] == 0; };
  int last_f[4] = {-1, -1, -1, -1};  // (warp 3) last chunk whose factors it copied, per slot

  if (warp < 4) {
    // ============================================================ chain
    for (int c = 0; c < nch; ++c) {
      const uint32_t s2 = c & 1, s4 = c & 3, p4 = (c >> 2) & 1;
      if (warp < 2) {  // D += A^T S^T: warp q takes K steps [8q, 8q + 8) into half q of cC slot s2
        wait(&bar_a[s4], p4);
        wait(&bar_b[s4], p4);
        tc_fence_after();
        if (live()) {
          const uint32_t dst = tmem + L::cC + s2 * 64 + (uint32_t)warp * SR;
          const uint32_t asrc = tmem + L::cA + s2 * 128 + (uint32_t)warp * 64;
          const uint64_t ds = dadd(dS32, (uint32_t)warp * 2u * (SR * 128));
          constexpr uint32_t idc = idesc_tf32(128, SR);
          auto f = [&](int j, bool) {
            if (elect_one()) mma_tf32_ts(dst, asrc + 8 * j, dadd(ds, (j >> 2) * (SR * 128) + (j & 3) * 32), idc, 1);
          };
          issue_range<0, 8>(f);
        }
        if (elect_one()) mma_commit(&bar_c[s4]);
        __syncwarp();
      }
      wait(&bar_f[s4], p4);
      const float gC = reinterpret_cast<const float*>(sm + L::FB + s4 * kFac)[63];
      wait(&bar_c[s4], p4);
      tc_fence_after();
      {  // S <- gamma_C S + D_hi + D_lo (lane = d_k)
        float dh[32], dl[32];
        tmem_ld32(tmem + lane_base + L::cC + s2 * 64, dh);
        tmem_ld32(tmem + lane_base + L::cC + s2 * 64 + SR, dl);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 d = __fadd2_rn(make_float2(dh[i], dh[i + 1]), make_float2(dl[i], dl[i + 1]));
          const float2 sn = __ffma2_rn(make_float2(gC, gC), make_float2(sreg[i], sreg[i + 1]), d);
          sreg[i] = sn.x;
          sreg[i + 1] = sn.y;
          *reinterpret_cast<float*>(sm + L::S32 + kf32(i, dcol, SR)) = tf32r(sn.x);
          *reinterpret_cast<float*>(sm + L::S32 + kf32(i + 1, dcol, SR)) = tf32r(sn.y);
        }
      }
      fence_async_smem();
      tc_fence_before();
      group_sync(1);  // the four chain warps: S^T complete for the next product, cC slot s2 read
      if (warp == 0 && elect_one()) mbar_arrive(&bar_s[s4]);
      // (warp 3) factors of chunk c + 4 into slot s4: the state update and U~s(c) have read them
      if (warp == 3 && lane == 0 && c + 4 < nch && live()) {
        load_f(c + 4);
        last_f[s4] = c + 4;
      }
      __syncwarp();
    }
  } else if (warp < 8) {
    // ============================================================ epilogues
    const int t = 32 * (quad & 1) + lane;  // token of this thread's lane (warps 4-5)
    for (int c = 0; c < nch; ++c) {
      const uint32_t s2 = c & 1, s4 = c & 3, p4 = (c >> 2) & 1;
      // Y(c) -> [Y_hi | Y_lo] (row d_k = this thread's lane), both truncated (|error| < 2^-15 |Y|)
      wait(&bar_y[s2], (c >> 1) & 1);
      if (c >= 2) wait(&bar_a[(c - 2) & 3], ((c - 2) >> 2) & 1);  // A^T(c-2) has read YS slot s2
      tc_fence_after();
      {
        float y0[32], y1[32];
        tmem_ld32(tmem + lane_base + L::cY, y0);
        tmem_ld32(tmem + lane_base + L::cY + 32, y1);
        tmem_ld_wait();
        tc_fence_before();
        unsigned char* ys = sm + L::YS + s2 * 32768;
        const uint32_t k = 32 * quad + lane;
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
          __align__(16) uint32_t hp[4], lp[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float a = i + e < 32 ? y0[i + e] : y1[i + e - 32];
            const float b = i + e + 1 < 32 ? y0[i + e + 1] : y1[i + e + 1 - 32];
            const float ha = hi16(a), hb = hi16(b);
            hp[e / 2] = bf16x2_trunc(ha, hb);
            lp[e / 2] = bf16x2_trunc(a - ha, b - hb);
          }
          *reinterpret_cast<uint4*>(ys + kbf16(k, i, 128)) = *reinterpret_cast<const uint4*>(hp);
          *reinterpret_cast<uint4*>(ys + kbf16(k, 64 + i, 128)) = *reinterpret_cast<const uint4*>(lp);
        }
        fence_async_smem();
        __syncwarp();
        if (elect_one()) mbar_arrive(&bar_ys[s4]);
        __syncwarp();
      }
      if (quad < 2) {  // U~s = diag(sc) U~ as bf16 hi + lo (token t), MN-major: hi in N [0, 32), lo in [32, 64)
        wait(&bar_u[s2], (c >> 1) & 1);
        if (c >= 2) wait(&bar_b[(c - 2) & 3], ((c - 2) >> 2) & 1);  // B^T(c-2) has read UH slot s2
        wait(&bar_f[s4], p4);
        tc_fence_after();
        float u[32];
        tmem_ld32(tmem + lane_base + L::cU + s2 * 32, u);
        tmem_ld_wait();
        tc_fence_before();
        const float sc = reinterpret_cast<const float*>(sm + L::FB + s4 * kFac)[64 + t];
        unsigned char* uh = sm + L::UH + s2 * 8192;
        __align__(16) uint32_t hp[16], lp[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float h0 = u[i] * sc, h1 = u[i + 1] * sc;
          const float t0 = hi16(h0), t1 = hi16(h1);
          hp[i / 2] = bf16x2_trunc(t0, t1);
          lp[i / 2] = bf16x2_trunc(h0 - t0, h1 - t1);
        }
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          *reinterpret_cast<uint4*>(uh + mnbf16(i, t, 64)) = *reinterpret_cast<const uint4*>(hp + i / 2);
          *reinterpret_cast<uint4*>(uh + mnbf16(SR + i, t, 64)) = *reinterpret_cast<const uint4*>(lp + i / 2);
        }
        fence_async_smem();
        __syncwarp();
        if (elect_one()) mbar_arrive(&bar_uh[s4]);
        __syncwarp();
      }
    }
  } else if (warp == 8) {
    // ============================================================ loads
    if (lane == 0) {
      int last_k[NKB] = {-1, -1, -1}, last_vr[2] = {-1, -1};
      for (int c = 0; c < min(nch, NKB); ++c) last_k[c % NKB] = c;
      for (int c = 0; c < min(nch, 2); ++c) last_vr[c & 1] = c;
      for (int c = 0; c < nch; ++c) {
        if (c + 2 < nch) {  // V and record part 1 of chunk c + 2 into slot c & 1: U~(c) and Y(c) read it
          wait(&bar_u[c & 1], (c >> 1) & 1);
          wait(&bar_y[c & 1], (c >> 1) & 1);
          if (live()) {
            load_vr(c + 2);
            last_vr[c & 1] = c + 2;
          }
        }
        if (c + NKB < nch) {  // K of chunk c + 3 into slot c % 3: Y(c), A^T(c) and B^T(c) read it
          wait(&bar_a[c & 3], (c >> 2) & 1);
          wait(&bar_b[c & 3], (c >> 2) & 1);
          if (live()) {
            load_k(c + NKB);
            last_k[c % NKB] = c + NKB;
          }
        }
      }
      // every copy issued into this CTA's shared memory has landed before the CTA may exit
      for (int s = 0; s < NKB; ++s)
        if (last_k[s] >= 0) mbar_wait(&bar_k[s], (uint32_t)(last_k[s] / NKB) & 1u, kDrainNs);
      for (int s = 0; s < 2; ++s)
        if (last_vr[s] >= 0) mbar_wait(&bar_vr[s], (uint32_t)(last_vr[s] >> 1) & 1u, kDrainNs);
    }
  } else {
    // ============================================================ MMA issuers
    const int role = warp - 9;  // 0: U~, 1: Y, 2: A^T, 3: B^T
    for (int c = 0; c < nch; ++c) {
      const uint32_t s2 = c & 1, s4 = c & 3, p4 = (c >> 2) & 1, kb = (uint32_t)(c % NKB);
      if (role == 0) {  // U~ = [Mb_hi | Mb_lo] [V; V] (M=128: rows 64-127 are not used)
        wait(&bar_vr[s2], (c >> 1) & 1);
        if (c >= 2) wait(&bar_uh[(c - 2) & 3], ((c - 2) >> 2) & 1);  // U~(c-2) read out of cU slot s2
        tc_fence_after();
        if (live()) {
          const uint64_t da = dadd(dMb, s2 * kRecPart1), db = dadd(dV, s2 * 8192);
          constexpr uint32_t id = idesc_bf16(128, SR, false, true);
          auto f = [&](int j, bool first) {
            if (elect_one())
              mma_bf16(tmem + L::cU + s2 * 32, dadd(da, (j >> 2) * 8192 + (j & 3) * 32), dadd(db, (j & 3) * 2048), id,
                       !first);
          };
          issue_range<0, 8>(f);
        }
        if (elect_one()) mma_commit(&bar_u[s2]);
      } else if (role == 1) {  // Y = K^T Z
        wait(&bar_k[kb], (uint32_t)(c / NKB) & 1u);
        wait(&bar_vr[s2], (c >> 1) & 1);
        if (c >= 1) wait(&bar_ys[(c - 1) & 3], ((c - 1) >> 2) & 1);  // Y(c-1) read out of cY
        tc_fence_after();
        if (live()) {
          const uint64_t da = dadd(dK, kb * 16384), db = dadd(dZ, s2 * kRecPart1);
          constexpr uint32_t id = idesc_bf16(128, 64, true, true);
          auto f = [&](int j, bool first) {
            if (elect_one()) mma_bf16(tmem + L::cY, dadd(da, j * 2048), dadd(db, j * 2048), id, !first);
          };
          issue_range<0, 4>(f);
        }
        if (elect_one()) mma_commit(&bar_y[s2]);
      } else if (role == 2) {  // A^T = [Y_hi | Y_lo] [K; K]
        wait(&bar_ys[s4], p4);
        if (c >= 2) wait(&bar_c[(c - 2) & 3], ((c - 2) >> 2) & 1);  // chain product c-2 read cA slot s2
        tc_fence_after();
        if (live()) {
          const uint64_t da = dadd(dYS, s2 * 32768), db = dadd(dK, kb * 16384);
          constexpr uint32_t id = idesc_bf16(128, 128, false, true);
          auto f = [&](int j, bool first) {
            if (elect_one())
              mma_bf16(tmem + L::cA + s2 * 128, dadd(da, (j >> 2) * 16384 + (j & 3) * 32), dadd(db, (j & 3) * 2048), id,
                       !first);
          };
          issue_range<0, 8>(f);
        }
        if (elect_one()) mma_commit(&bar_a[s4]);
      } else {  // B^T = K^T [U~s_hi | U~s_lo]
        wait(&bar_uh[s4], p4);
        if (c >= 2) wait(&bar_s[(c - 2) & 3], ((c - 2) >> 2) & 1);  // state update c-2 read cC slot s2
        tc_fence_after();
        if (live()) {
          const uint64_t da = dadd(dK, kb * 16384), db = dadd(dUH, s2 * 8192);
          constexpr uint32_t id = idesc_bf16(128, 64, true, true);
          auto f = [&](int j, bool first) {
            if (elect_one()) mma_bf16(tmem + L::cC + s2 * 64, dadd(da, j * 2048), dadd(db, j * 2048), id, !first);
          };
          issue_range<0, 4>(f);
        }
        if (elect_one()) mma_commit(&bar_b[s4]);
      }
      __syncwarp();
    }
  }

  // Drain: every issuing warp's products have completed, and the factor copies have landed,
  // before TMEM is freed and the CTA exits.
  if (warp == 0 || warp == 1 || warp >= 9) {
    if (elect_one()) mma_commit(bar_dr);
    __syncwarp();
  }
  if (warp == 3 && lane == 0)
    for (int s = 0; s < 4; ++s)
      if (last_f[s] >= 0) mbar_wait(&bar_f[s], (uint32_t)(last_f[s] >> 2) & 1u, kDrainNs);
  __syncthreads();
  if (tid == 0 && !mbar_wait(bar_dr, 0, kDrainNs)) flags[0] = 1;
  __syncthreads();
  if (flags[0]) {
    if (tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);
  } else if (warp < 4) {
#pragma unroll
    for (int r = 0; r < SR; ++r) p.S_out[sbase + (size_t)(row0 + r) * DK + dcol] = sreg[r];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace

cudaError_t launch_state_tc(const CUtensorMap& mk, const CUtensorMap& mv, const StateParams& sp, bool overlap_prep,
                            cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)StLay::ALLOC);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the prep kernel, as the scan (see launch_scan)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(DV / SR, sp.h_v, sp.n_seqs);
  cfg.blockDim = dim3(SNT);
  cfg.dynamicSmemBytes = StLay::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap_prep ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_state_kernel, mk, mv, sp);
}

}  // namespace gdn
