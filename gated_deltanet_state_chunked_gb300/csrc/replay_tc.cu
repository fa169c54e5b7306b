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
// Kernels:
//  * chunk_prep_kernel -- the (chunk, key head) items of all tails, walked by a persistent
//    grid of two CTAs per SM: K K^T on tcgen05, the gated A and P, and M = (I + A)^{-1}
//    (16x16 diagonal blocks by forward substitution on CUDA cores, then two levels of block
//    merges on warp-level tensor cores), written with beta, G and rk to a per-(chunk, v-head)
//    record in scratch memory.
//  * tail_order_kernel -- with several tails, their order longest first.
//  * chunk_scan_kernel -- one CTA per 32- or 64-row slice of d_v of one (tail, v-head)
//    state, walking the tail's chunks (R = 32 while all slices fit on the GPU at once, else
//    64).  Per chunk:
//      W = Mw K           bf16 (computed factor rounded once)            M=128 N=128 K=64
//      [Mb_hi|Mb_lo][V;V] bf16 hi/lo split of the computed factor        M=128 N=R   K=128
//      [W;Q] S0^T         tf32, [W;Q] from TMEM (W truncated to tf32     M=128 N=R   K=128
//                         by the read, S0 rounded to nearest, Q exact)
//      K^T U^             bf16 split of the scaled U: with 32-row slices
//                         [K^T U^hi | K^T U^lo], two warps over 32 tokens  M=128 N=2R  K=32 each;
//                         with 64-row slices [K^T|K^T][U^hi;U^lo]         M=128 N=R   K=128
//      P U                tf32                                           M=128 N=R   K=64
//    (the M=128 shapes with 64 meaningful rows put them where the epilogue needs them)
//    all accumulated in fp32 in TMEM; the state slice stays in fp32 registers.
// State-only calls with 32-row slices take the operator-form scan of state_tc.cu instead; the
// prep kernel then stores Z = -diag(rk exp(G_last - G)) Mw in Mw's place.
// Padded tokens past a tail's end get beta = g = 0 (identity transitions).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
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
// Inside one chunk the gate sums span fewer binades than this in all but extreme inputs; then
// exp2(G_t - G_s) is evaluated as exp2(G_t - G_last) * exp2(G_last - G_s) without leaving the
// fp32 range, else per element.
constexpr float kFactorRange = 100.f;

struct PrepLay {
  static constexpr uint32_t KQ = 0;                      // bf16 [K;Q]: 2 d_k atoms x (128 rows x 128 B)
  static constexpr uint32_t SLOT = 32768;                // two v-head slots:
  static constexpr uint32_t AMAT = 0;                    //   fp32 64 x 68 (A, then block scratch)
  static constexpr uint32_t MMAT = 64 * MST * 4;         //   fp32 64 x 68 (M)
  static constexpr uint32_t GATE = 2 * 64 * MST * 4;     //   8 x 64 floats
  static constexpr uint32_t SLOT_BYTES = GATE + 2048;
  static constexpr uint32_t COMMON = SLOT + 2 * SLOT_BYTES;  // rk[64], rq[64]
  static constexpr uint32_t BARS = COMMON + 512;
  static constexpr uint32_t TOTAL = BARS + 128;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
};

struct PrepParams {
  const float* g;
  const float* beta;
  const int32_t* cu;
  unsigned char* rec;  // records [chunk][h_v]
  int* status;
  int n_seqs, total_tokens, h_k, h_v, l2norm, write_O;
  int scalar_decay;  // 1: A = 0 (M = I) and W = 0 (no rank-1 projection term)
  int zform;         // 1: store Z = -diag(rk exp(G_last - G)) Mw in place of Mw (operator-form scan)
  float scale;
};

// Row sum of squares of a 64-element bf16 row held as 8 16-byte chunks (any order).
__device__ __forceinline__ float row_sumsq(const unsigned char* row, int rot) {
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = reinterpret_cast<const uint4*>(row)[(c + rot) & 7];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
  return ss;
}

__global__ void __launch_bounds__(NT, 2) chunk_prep_kernel(const __grid_constant__ CUtensorMap map_q,
                                                           const __grid_constant__ CUtensorMap map_k, PrepParams p) {
  using L = PrepLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* cRk = reinterpret_cast<float*>(sm + L::COMMON);
  float* cRq = cRk + 64;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 16);
  int* fact = reinterpret_cast<int*>(sm + L::BARS + 24);  // [2], per slot
  int* scratch = reinterpret_cast<int*>(sm + L::BARS + 32);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, half = warp >> 2;
  const int G = p.h_v / p.h_k;
  grid_dep_launch();  // the scan may start launching once every prep CTA is running
  // Work items (chunk, key head), item = chunk * h_k + key head, strided over a grid of about
  // two CTAs per SM.  While a CTA works on one item it fetches the next one's gates and, once
  // this item's P has left the [K;Q] area, its K and Q tiles.
  struct Item {
    int gc, hk, t0, n;
    bool ok;
  };
  int total = 0;
  auto item_at = [&](int item) {  // block-wide (chunk_info synchronises the CTA)
    Item r;
    r.gc = item / p.h_k;
    r.hk = item - r.gc * p.h_k;
    const ChunkInfo ci = chunk_info(p.cu, p.n_seqs, p.total_tokens, -1, r.gc, scratch);
    total = ci.total;
    r.ok = r.gc < ci.total && ci.gc_seq >= 0;
    r.t0 = r.ok ? p.cu[ci.gc_seq] + ci.gc_idx * C : 0;
    r.n = r.ok ? min(C, p.cu[ci.gc_seq + 1] - r.t0) : 0;
    return r;
  };
  // g and beta of an item's first slot pair (warp 0 of each warpgroup: tokens lane and lane + 32
  // of its slot)
  auto load_gb = [&](const Item& it, float (&pre)[4]) {
    pre[0] = pre[1] = pre[2] = pre[3] = 0.f;
    if (it.ok && (warp & 3) == 0 && half < min(2, G)) {
      const int h = it.hk * G + half;
      if (lane < it.n) {
        pre[0] = p.g[(size_t)(it.t0 + lane) * p.h_v + h];
        pre[2] = p.beta[(size_t)(it.t0 + lane) * p.h_v + h];
      }
      if (lane + 32 < it.n) {
        pre[1] = p.g[(size_t)(it.t0 + lane + 32) * p.h_v + h];
        pre[3] = p.beta[(size_t)(it.t0 + lane + 32) * p.h_v + h];
      }
    }
  };
  auto issue_tma = [&](const Item& it) {  // one thread
    mbar_arrive_expect_tx(bar_tma, 32768);
    for (int a = 0; a < 2; ++a) {
      tma_load_2d(sm + L::KQ + a * 16384, &map_k, bar_tma, it.hk * DK + a * 64, it.t0);
      tma_load_2d(sm + L::KQ + a * 16384 + 8192, &map_q, bar_tma, it.hk * DK + a * 64, it.t0);
    }
  };
  Item cur = item_at(blockIdx.x);
  const int n_items = total * p.h_k;
  if ((int)blockIdx.x >= n_items) return;
  float pre[4];
  load_gb(cur, pre);

  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    if (cur.ok) issue_tma(cur);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Gate sums of a slot (warp 0 of its warpgroup; tokens lane and lane + 32): inclusive sums G
  // in log2 units, exp2(G - G_last) and exp2(G_last - G).  For the first pair they are formed
  // here, while the K, Q tiles are in flight.
  struct GateSums {
    float la, lb, ea, eb, fa, fb, ba, bb;
  };
  auto gate_sums = [&](float ga, float gb, float ba, float bb) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float xa = __shfl_up_sync(0xffffffffu, ga, o);
      const float xb = __shfl_up_sync(0xffffffffu, gb, o);
      if (lane >= o) { ga += xa; gb += xb; }
    }
    gb += __shfl_sync(0xffffffffu, ga, 31);
    GateSums r;
    r.la = ga * kLog2e;
    r.lb = gb * kLog2e;
    const float last = __shfl_sync(0xffffffffu, r.lb, 31);
    r.ea = exp2f(r.la - last); r.eb = exp2f(r.lb - last);
    r.fa = exp2f(last - r.la); r.fb = exp2f(last - r.lb);
    r.ba = ba; r.bb = bb;
    return r;
  };
  int done = 0;  // items processed: the parity of bar_tma and bar_mma
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int gc = cur.gc, hk = cur.hk, t0 = cur.t0, n = cur.n;
    Item nxt{0, 0, 0, 0, false};
    if (item + (int)gridDim.x < n_items) nxt = item_at(item + gridDim.x);  // uniform
    float pre_n[4];
    load_gb(nxt, pre_n);  // in flight during this item
    if (!cur.ok) {  // (not reached for well-formed offsets) nothing was fetched for this item
      cur = nxt;
#pragma unroll
      for (int i = 0; i < 4; ++i) pre[i] = pre_n[i];
      if (tid == 0 && cur.ok) issue_tma(cur);
      continue;
    }
    const uint32_t ph = (uint32_t)(done & 1);
    GateSums gs0 = {};
    if ((warp & 3) == 0 && half < min(2, G)) gs0 = gate_sums(pre[0], pre[1], pre[2], pre[3]);
    bool ok = mbar_wait(bar_tma, ph, kWaitNs);
    if (tid == 0) {
      tc_fence_after();  // the previous item's Gram has been read out of TMEM by every thread
      const uint64_t d = sdesc_sw128(smem_u32(sm + L::KQ), 16, 1024);
      constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t dj = d + (uint64_t)((((j >> 2) * 16384) + (j & 3) * 32) >> 4);
        mma_bf16(tmem, dj, dj, id, j > 0);
      }
      mma_commit(bar_mma);
    }
    {  // norms: 128 rows (64 keys, 64 queries) x 2 atoms, rotated chunk order (no bank conflicts)
      const int row = tid >> 1, atom = tid & 1;
      float ss = row_sumsq(sm + L::KQ + atom * 16384 + row * 128, row);
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (atom == 0) {
        const float r = p.l2norm ? 1.f / sqrtf(ss + 1e-6f) : 1.f;
        if (row < 64) cRk[row] = r;
        else cRq[row - 64] = r * p.scale;
      }
    }
    ok = mbar_wait(bar_mma, ph, kWaitNs) && ok;
    tc_fence_after();
    float kq[32];  // row (32*quad + lane) of [K;Q] K^T, columns [32*half, +32)
    tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + half * 32, kq);
    tmem_ld_wait();
    tc_fence_before();
    if (!ok && tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);
    __syncthreads();

    const int slot = half, gt = tid & 127;  // warpgroup = v-head slot
    unsigned char* sslot = sm + L::SLOT + slot * L::SLOT_BYTES;
    float* amat = reinterpret_cast<float*>(sslot + L::AMAT);
    float* mmat = reinterpret_cast<float*>(sslot + L::MMAT);
    float* gB = reinterpret_cast<float*>(sslot + L::GATE);  // beta
    float* gG2 = gB + 64;   // G log2(e)
    float* gFa = gB + 128;  // beta_t rk_t exp2(G_t - G_last)
    float* gFc = gB + 192;  // rk_s exp2(G_last - G_s)
    float* gPa = gB + 256;  // rq_t exp2(G_t - G_last)
    float* gGam = gB + 320; // gamma_t

    for (int pair = 0; pair < G; pair += 2) {
      const int nslots = min(2, G - pair);
      // gates of both slots: warp 0 of each warpgroup
      if ((warp & 3) == 0 && slot < nslots) {
        const int h = hk * G + pair + slot;
        GateSums q = gs0;
        if (pair > 0) {
          const float ga = lane < n ? p.g[(size_t)(t0 + lane) * p.h_v + h] : 0.f;
          const float gb = lane + 32 < n ? p.g[(size_t)(t0 + lane + 32) * p.h_v + h] : 0.f;
          const float ba = lane < n ? p.beta[(size_t)(t0 + lane) * p.h_v + h] : 0.f;
          const float bb = lane + 32 < n ? p.beta[(size_t)(t0 + lane + 32) * p.h_v + h] : 0.f;
          q = gate_sums(ga, gb, ba, bb);
        }
        const float la = q.la, lb = q.lb, ea = q.ea, eb = q.eb, fa = q.fa, fb = q.fb, ba = q.ba, bb = q.bb;
        const float last = __shfl_sync(0xffffffffu, lb, 31);
        gB[lane] = ba; gB[lane + 32] = bb;
        gG2[lane] = la; gG2[lane + 32] = lb;
        gFa[lane] = ba * cRk[lane] * ea; gFa[lane + 32] = bb * cRk[lane + 32] * eb;
        gFc[lane] = cRk[lane] * fa; gFc[lane + 32] = cRk[lane + 32] * fb;
        gPa[lane] = cRq[lane] * ea; gPa[lane + 32] = cRq[lane + 32] * eb;
        gGam[lane] = exp2f(la); gGam[lane + 32] = exp2f(lb);
        if (lane == 0) fact[slot] = (la - last) < kFactorRange ? 1 : 0;
      }
      __syncthreads();
      // A (key rows) and P (query rows) for each slot from this thread's Gram row
      {
        const int row = 32 * quad + lane;
        for (int sl = 0; sl < nslots; ++sl) {
          unsigned char* ss_ = sm + L::SLOT + sl * L::SLOT_BYTES;
          float* A_ = reinterpret_cast<float*>(ss_ + L::AMAT);
          const float* B_ = reinterpret_cast<const float*>(ss_ + L::GATE);
          const float *G2_ = B_ + 64, *Fa_ = B_ + 128, *Fc_ = B_ + 192, *Pa_ = B_ + 256;
          if (row < 64) {
            const int t = row;
            float av[32];
            if (fact[sl]) {
              // (at Fc_s) kq in packed pairs; the 32x32 block of this warp's rows and columns is
              // below, on or above the diagonal as a whole (warp-uniform), masked only on it
              const int rel = quad - half;
              const float at = Fa_[t];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 f = *reinterpret_cast<const float2*>(Fc_ + half * 32 + i);
                const float2 x = __fmul2_rn(__fmul2_rn(make_float2(at, at), f), make_float2(kq[i], kq[i + 1]));
                av[i] = rel < 0 ? 0.f : x.x;
                av[i + 1] = rel < 0 ? 0.f : x.y;
              }
              if (rel == 0) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (half * 32 + i >= t) av[i] = 0.f;
              }
            } else {
              const float bt = B_[t] * cRk[t], g_t = G2_[t];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int s = half * 32 + i;
                av[i] = s < t ? bt * exp2f(g_t - G2_[s]) * cRk[s] * kq[i] : 0.f;
              }
            }
            if (p.scalar_decay) {  // scalar-decay family: no rank-1 projection, A = 0 and M = I
#pragma unroll
              for (int i = 0; i < 32; ++i) av[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(A_ + t * MST + half * 32 + i) = make_float4(av[i], av[i + 1], av[i + 2], av[i + 3]);
          } else if (p.write_O) {
            const int t = row - 64;
            // staged in the record's own layout in the [K;Q] area (free once the Gram and the norms
            // have read it), 16 KB per slot, then stored by one bulk copy
            unsigned char* Pst = sm + L::KQ + sl * 16384;
            float x[32];
            if (fact[sl]) {
              const int rel = quad - 2 - half;
              const float at = Pa_[t];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 f = *reinterpret_cast<const float2*>(Fc_ + half * 32 + i);
                const float2 y = __fmul2_rn(__fmul2_rn(make_float2(at, at), f), make_float2(kq[i], kq[i + 1]));
                x[i] = rel < 0 ? 0.f : tf32r(y.x);
                x[i + 1] = rel < 0 ? 0.f : tf32r(y.y);
              }
              if (rel == 0) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (half * 32 + i > t) x[i] = 0.f;
              }
            } else {
              const float qt = cRq[t], g_t = G2_[t];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int s = half * 32 + i;
                x[i] = s <= t ? tf32r(qt * exp2f(g_t - G2_[s]) * cRk[s] * kq[i]) : 0.f;
              }
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(Pst + kf32(t, half * 32 + i, 64)) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
          }
        }
      }
      fence_async_smem();  // the staged P -> the bulk copy
      __syncthreads();
      // P to the records: a 16 KB bulk copy per slot, in flight during the inverse.  Issued by a
      // thread of warp 3 of slot 0, which only clears M's upper blocks before the inverse's first
      // barrier (issuing can hold a thread for about a thousand cycles).
      const bool issP = p.write_O && tid == 96;
      if (issP) {
        for (int sl = 0; sl < nslots; ++sl) {
          const int h = hk * G + pair + sl;
          bulk_store(p.rec + ((size_t)gc * p.h_v + h) * kRecBytes + kRecP, sm + L::KQ + sl * 16384, 16384);
        }
        bulk_commit();
      }
      if (slot < nslots) {
        invert_unit_lower(amat, mmat, gt, 1 + slot);
        if (tid == 96 && pair + 2 >= G && nxt.ok) {  // the next item's K and Q tiles: the [K;Q]
          if (p.write_O) bulk_wait_read_all();       // area is free once the P copies have read it
          issue_tma(nxt);
        }
        // record: Mb hi|lo, Mw, per-token factors
        const int h = hk * G + pair + slot;
        unsigned char* rec = p.rec + ((size_t)gc * p.h_v + h) * kRecBytes;
        // item (row t, columns [s, s + 8)): a quarter-warp writes whole 128-byte rows; the
        // column factors are the same for all four rows of a thread
        const int s = 8 * (gt & 7);
        const float4 b0 = *reinterpret_cast<const float4*>(gB + s), b1 = *reinterpret_cast<const float4*>(gB + s + 4);
        const float4 y0 = *reinterpret_cast<const float4*>(gGam + s), y1 = *reinterpret_cast<const float4*>(gGam + s + 4);
        const float4 r0 = *reinterpret_cast<const float4*>(cRk + s), r1 = *reinterpret_cast<const float4*>(cRk + s + 4);
        // Mw = M diag(beta gamma rk); zero for the scalar-decay family (no correction W S0^T)
        const float wz = p.scalar_decay ? 0.f : 1.f;
        const float wf[8] = {wz * y0.x * r0.x, wz * y0.y * r0.y, wz * y0.z * r0.z, wz * y0.w * r0.w,
                             wz * y1.x * r1.x, wz * y1.y * r1.y, wz * y1.z * r1.z, wz * y1.w * r1.w};
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int t = 16 * it + (gt >> 3);
          const float4 m0 = *reinterpret_cast<const float4*>(mmat + t * MST + s);
          const float4 m1 = *reinterpret_cast<const float4*>(mmat + t * MST + s + 4);
          const float mb[8] = {m0.x * b0.x, m0.y * b0.y, m0.z * b0.z, m0.w * b0.w,
                               m1.x * b1.x, m1.y * b1.y, m1.z * b1.z, m1.w * b1.w};
          const float zt = p.zform ? -gFc[t] : 1.f;  // row factor of Z
          __align__(16) uint32_t bh[4], bl[4], wv[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            // Mb as bf16 hi + lo, both truncated (|error| < 2^-15 |Mb|); Mw rounded to nearest even
            const float h0 = __uint_as_float(__float_as_uint(mb[e]) & 0xffff0000u);
            const float h1 = __uint_as_float(__float_as_uint(mb[e + 1]) & 0xffff0000u);
            bh[e / 2] = bf16x2_trunc(h0, h1);
            bl[e / 2] = bf16x2_trunc(mb[e] - h0, mb[e + 1] - h1);
            wv[e / 2] = bf16x2_rne(mb[e] * wf[e] * zt, mb[e + 1] * wf[e + 1] * zt);
          }
          *reinterpret_cast<uint4*>(rec + kRecMB + kbf16(t, s, 64)) = *reinterpret_cast<const uint4*>(bh);
          *reinterpret_cast<uint4*>(rec + kRecMB + kbf16(t, 64 + s, 64)) = *reinterpret_cast<const uint4*>(bl);
          *reinterpret_cast<uint4*>(rec + kRecMW + kbf16(t, s, 64)) = *reinterpret_cast<const uint4*>(wv);
        }
        if (gt < 64) {
          float* gate = reinterpret_cast<float*>(rec + kRecGate);
          gate[gt] = gGam[gt];
          gate[64 + gt] = gFc[gt];
          gate[128 + gt] = gGam[gt] * cRq[gt];
        }
      }
      if (issP) bulk_wait_read_all();  // the next pair restages P; the source stays until read
      __syncthreads();
    }
    ++done;
    cur = nxt;
#pragma unroll
    for (int i = 0; i < 4; ++i) pre[i] = pre_n[i];
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
  // 32-row slices (the latency case, few problems): every tile a chunk needs is requested a
  // whole chunk ahead (K has three buffers, Q two), M diag(beta) and P are A operands in TMEM
  // (a 64-column region shared by both: Mb in lanes 0-63, P in lanes 64-127; each product's
  // other 64 rows are results nobody reads), and K^T [U^hi | U^lo] has N = 2R (K^T read once),
  // split over two warps by tokens.  64-row slices (the throughput case) have no TMEM columns to spare:
  // Mb and P are read from shared memory, K and Q are copied once the chain has finished the
  // chunk two before (two K buffers, one Q), and K^T U^ runs over K = [tokens; tokens].
  static constexpr bool NARROW = R == 32;
  static constexpr bool EARLY_KQ = NARROW;
  static constexpr int NKB = EARLY_KQ ? 3 : 2, NQB = EARLY_KQ ? 2 : 1;
  static constexpr uint32_t KB = 0;                 // NKB buffers of bf16 K: 2 d_k atoms x (64 rows x 128 B)
  static constexpr uint32_t QB = KB + NKB * 16384;  // NQB buffers of bf16 Q: 2 d_k atoms x (64 rows x 128 B)
  static constexpr uint32_t VT = QB + NQB * 16384;  // bf16 V atom: 64 tokens x 128 B
  static constexpr uint32_t R1 = VT + 8192;         // record part 1: Mb hi|lo (16 KB), Mw (8 KB)
  static constexpr uint32_t R2 = R1 + kRecPart1;    // 2 buffers of record part 2: P (16 KB), factors (1 KB)
  static constexpr uint32_t UH = R2 + 2 * 18432;    // bf16 U^ hi and lo, MN-major (see the U epilogue)
  static constexpr uint32_t UT = UH + 16384;        // fp32 U^T (R rows x 2 atoms)
  static constexpr uint32_t S32 = UT + R * 256;     // fp32 state slice (R rows x 4 atoms), tf32-rounded
  static constexpr uint32_t BARS = S32 + R * 512;
  static constexpr uint32_t TOTAL = BARS + 256;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM columns.  All accumulators use the M=128 layout (lane = row).  cWQ holds the fp32
  // [W;Q] operand of [W;Q] S0^T (lane = token row, column = d_k), read by the MMA straight from
  // TMEM (as tf32: the low mantissa bits of W are dropped, Q is exact).  [W;Q] S0^T and U~ put
  // the chunk's tokens in lanes 0-63 (W S0^T, U~) and 64-127 (Q S0^T; P U is aimed there too).
  // U~ and [W;Q] S0^T have one copy per chunk parity: a chunk's outputs are read back while the
  // next chunk's [W;Q] S0^T runs.  P U has one copy: the next P U is issued only after the
  // outputs have read it.  [W;Q] S0^T and P U are each issued by one warp; with 32-row slices
  // K^T U^ comes from the two warps that wrote the U^ rows, each over its own 32 tokens.
  static constexpr int ND1 = 1, NPU = 1;
  // K^T U^: 32-row slices two accumulators of 2R columns ([hi | lo]), one per issuing warp (each
  // covers the 32 tokens whose U^ rows that warp wrote); 64-row slices one of R columns
  static constexpr int ND2 = NARROW ? 2 : 1;
  static constexpr uint32_t D2COLS = NARROW ? 4 * R : R;
  // accumulator a of [W;Q] S0^T for chunk parity b: cD1 + (2 a + b) R; of P U: cPU + a R
  static constexpr uint32_t cWQ = 0, cU = 128, cD1 = 128 + 2 * R, cD2 = cD1 + 2 * R * ND1, cPU = cD2 + D2COLS;
  static constexpr uint32_t cMP = cPU + R * NPU;  // (32-row slices) Mb in lanes 0-63, P in lanes 64-127
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(cMP + (NARROW ? 64 : 0) <= TMEM_COLS, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(QB % 1024 == 0 && R2 % 1024 == 0 && UH % 1024 == 0 && UT % 1024 == 0 &&
                    S32 % 1024 == 0 && R1 >= 8192,
                "tile alignment");
};

struct ScanParams {
  const int32_t* cu;
  const int32_t* order;  // tails longest first (scan CTA z takes tail order[z]), or null
  const float* S0;
  const unsigned char* rec;
  __nv_bfloat16* O;
  float* S_out;
  int* status;
  int n_seqs, total_tokens, h_k, h_v;
  int write_O;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}


// Advance a shared-memory descriptor's start address by a byte offset (multiple of 16).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// f(j, j == J0) for j = J0 .. J1-1, unrolled at compile time (an MMA issue loop whose operand
// offsets fold to constants).  Issue sites run on a whole converged warp with warp-uniform
// operands; f issues through elect_one().
template <int J0, int J1, typename F>
__device__ __forceinline__ void issue_range(F&& f) {
#pragma unroll
  for (int j = J0; j < J1; ++j) f(j, j == J0);
}

// Warp-specialised scan.  Warps 0-3 ("chain") carry the state from chunk to chunk:
//   D1 = [W;Q] S0^T -> U = U~ - W S0^T, U^ -> D2 = K^T U^ (state), P U (outputs) -> S = gamma_C S + D2.
// Warps 0-1 form U from the token rows 0-63 of D1 while warps 2-3 write the previous chunk's
// outputs from rows 64-127 (Q S0^T) and P U, so the output epilogue is off the chunk-to-chunk
// chain.  Warps 4-7 ("prep") run one chunk ahead: the W = Mw K and U~ MMAs, the [W;Q]
// operand in TMEM (the Q rows stored beside W), with 32-row slices Mb and P in TMEM, and all
// loads.  The groups hand over through mbarriers that complete once per chunk.
template <int R>
__global__ void __launch_bounds__(NT, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, ScanParams p) {
  using L = ScanLay<R>;
  static_assert(R == 32 || R == 64, "state slices of 32 or 64 rows per CTA");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_kq = bars + 0;   // [2] loads of K and Q
  uint64_t* bar_r2 = bars + 2;   // [2] loads of record part 2
  uint64_t* bar_r1 = bars + 4;   // V + record part 1
  uint64_t* bar_w = bars + 5;    // MMA W = Mw K
  uint64_t* bar_u = bars + 6;    // MMA U~
  uint64_t* bar_d1 = bars + 7;   // MMA [W;Q] S0^T
  uint64_t* bar_d2 = bars + 8;   // MMA K^T U^
  uint64_t* bar_pu = bars + 9;   // MMA P U
  constexpr int NBARS = 10;
  // Hand-offs between the two warp groups are named barriers (an mbarrier hand-off between warps
  // of one SM costs about 200 cycles, a named barrier about 36).  Each is arrived at by one group
  // and synchronised on by the other, once per chunk, and every use strictly alternates with the
  // other side's, by construction (so counts never mix and neither side can wait forever on an
  // arrival that the other made for a different chunk):
  //   NB_W  prep -> chain: [W;Q], U~ (and Mb) of chunk c are in TMEM.  The prep arrives for chunk
  //         c only after NB_S of chunk c-1, which the chain arrives at after it synchronised
  //         on NB_W of chunk c-1.
  //   NB_S  chain -> prep: chunk c is finished (its P U has completed, its factors were read).
  //         The chain arrives for chunk c+1 only after NB_W of chunk c+1.
  //   NB_P  prep (warps 6-7) -> the P U issuer (warp 1), 32-row slices with outputs: P of chunk
  //         c is in TMEM.  Arrived at after NB_S of chunk c-1; synchronised on before P U of c,
  //         which precedes the chain's NB_S of chunk c.  (64 + 32 threads.)
  constexpr int NB_W = 3, NB_S = 4, NB_P = 5;
  // buffers of chunk c's K and Q tiles
  auto kbuf = [&](int c) { return (uint32_t)(c % L::NKB); };
  auto qbuf = [&](int c) { return (uint32_t)(L::NQB == 2 ? c & 1 : 0); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 128);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + L::BARS + 132);
  int* scratch = reinterpret_cast<int*>(sm + L::BARS + 160);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const bool chain = warp < 4;
  const int slice = blockIdx.x, h = blockIdx.y, seq = p.order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int row0 = slice * R;
  const int hk = h / (p.h_v / p.h_k);

  // A malformed range (see chunk_info) has no records: report it before forming any address.
  const ChunkInfo ci = chunk_info(p.cu, p.n_seqs, p.total_tokens, seq, -1, scratch);
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
  auto load_kq = [&](int c) {
    const int b = c & 1, t0c = t_begin + c * C;
    mbar_arrive_expect_tx(&bar_kq[b], 32768);
    for (int a = 0; a < 2; ++a) {
      tma_load_2d(sm + L::KB + kbuf(c) * 16384 + a * 8192, &map_k, &bar_kq[b], hk * DK + a * 64, t0c);
      tma_load_2d(sm + L::QB + qbuf(c) * 16384 + a * 8192, &map_q, &bar_kq[b], hk * DK + a * 64, t0c);
    }
  };
  auto load_r2 = [&](int c) {
    const int b = c & 1;
    mbar_arrive_expect_tx(&bar_r2[b], kRecPart2);
    bulk_load(sm + L::R2 + b * 18432, rec_of(c) + kRecPart1, kRecPart2, &bar_r2[b]);
  };
  auto load_r1 = [&](int c) {
    mbar_arrive_expect_tx(bar_r1, 8192 + kRecPart1);
    tma_load_2d(sm + L::VT, &map_v, bar_r1, h * DV + (row0 & ~63), t_begin + c * C);
    bulk_load(sm + L::R1, rec_of(c), kRecPart1, bar_r1);
  };
  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {  // the MMA barriers count one commit per issuing warp
      const int n = &bars[i] == bar_d1 ? L::ND1 : &bars[i] == bar_pu ? L::NPU : &bars[i] == bar_d2 ? L::ND2 : 1;
      mbar_init(&bars[i], n);
    }
    mbar_fence_init();
    flags[0] = 0;
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    if (nch > 0) load_kq(0);
    grid_dep_wait();  // the records are written by the prep kernel
    if (nch > 0) {
      load_r1(0);
      load_r2(0);
    }
    if (nch > 1) load_r2(1);
  }
  grid_dep_wait();

  // entering state (chain warps): thread owns d = 32*quad + lane and all R columns, fp32 registers
  const int dcol = 32 * quad + lane;
  float sreg[R];
  const size_t sbase = ((size_t)seq * p.h_v + h) * DV * DK;
  if (chain) {
#pragma unroll
    for (int c = 0; c < R; ++c) {
      const float s = p.S0 ? p.S0[sbase + (size_t)(row0 + c) * DK + dcol] : 0.f;
      sreg[c] = s;
      *reinterpret_cast<float*>(sm + L::S32 + kf32(c, dcol, R)) = tf32r(s);
    }
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t vcoloff = (uint32_t)(row0 & 63) * 2u;
  const uint64_t dKmn = sdesc_sw128(smem_u32(sm + L::KB), 8192, 1024);  // MN-major view of K
  const uint64_t dVT = sdesc_sw128(smem_u32(sm + L::VT) + vcoloff, 8192, 1024);
  const uint64_t dR1 = sdesc_sw128(smem_u32(sm + L::R1), 16, 1024);
  // P as rows 64-127 of an M=128 operand: the view starts 64 rows (8 KB) before each P buffer
  const uint64_t dR2p = sdesc_sw128(smem_u32(sm + L::R2 - 8192), 16, 1024);
  const uint64_t dUHmn = sdesc_sw128(smem_u32(sm + L::UH), 16384, 1024);
  const uint64_t dUT = sdesc_sw128(smem_u32(sm + L::UT), 16, 1024);
  const uint64_t dS32 = sdesc_sw128(smem_u32(sm + L::S32), 16, 1024);
  // Bounded wait.  After the first timeout every later wait returns at once, so both
  // warp groups run their (uniform) loops to the end and the CTA exits with an error.  Every wait
  // suspends rather than polls: a polling warp takes issue slots from the warps that share its
  // scheduler (measured: polling chain warps cost 1.6 us per 3277-token call).
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (flags[0]) return;
    if (!mbar_wait(bar, parity, kWaitNs)) flags[0] = 1;
  };

  if (chain) {
    // ============================================================ chain warps
    const int t = 32 * (quad & 1) + lane;  // token of this thread's TMEM lane (lane 32*quad + lane)
    float gq_prev = 0.f;                   // output gate of token t in the previous chunk (warps 2-3)
    // warps 2-3: O of chunk cc = gq (Q S0^T) + P U, from rows 64-127 of cc's accumulators
    auto outputs = [&](int cc) {
      const uint32_t pb = (uint32_t)(cc & 1) * R;
      const int t0c = t_begin + cc * C, n = min(C, t_end - t0c);
      wait(bar_pu, (uint32_t)(cc & 1));  // P U of chunk cc
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < R / 32; ++hh) {  // 32 state rows at a time
        float dq[32], pu[32];
        tmem_ld32(tmem + lane_base + L::cD1 + pb + 32 * hh, dq);
        tmem_ld32(tmem + lane_base + L::cPU + 32 * hh, pu);
        tmem_ld_wait();
#pragma unroll
        for (int a = 1; a < L::ND1; ++a) {
          float x[32];
          tmem_ld32(tmem + lane_base + L::cD1 + (2 * a) * R + pb + 32 * hh, x);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) dq[i] += x[i];
        }
#pragma unroll
        for (int a = 1; a < L::NPU; ++a) {
          float x[32];
          tmem_ld32(tmem + lane_base + L::cPU + a * R + 32 * hh, x);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) pu[i] += x[i];
        }
        if (t < n) {
          __align__(16) __nv_bfloat162 o[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            o[i / 2] = __floats2bfloat162_rn(fmaf(gq_prev, dq[i], pu[i]), fmaf(gq_prev, dq[i + 1], pu[i + 1]));
          __nv_bfloat16* dst = p.O + ((size_t)(t0c + t) * p.h_v + h) * DV + row0 + 32 * hh;
#pragma unroll
          for (int i = 0; i < 32; i += 8)
            *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<const uint4*>(o + i / 2);
        }
      }
    };
    for (int c = 0; c < nch; ++c) {
      const uint32_t par = c & 1;
      const float* gate = reinterpret_cast<const float*>(sm + L::R2 + par * 18432 + (kRecGate - kRecPart1));
      named_sync(NB_W, 256);
      if (warp < L::ND1) {  // D1 = [W;Q] S0^T (tf32, [W;Q] from TMEM: 8 columns per K step)
        tc_fence_after();
        constexpr uint32_t id1 = idesc_tf32(128, R);
        const uint32_t dst = tmem + L::cD1 + (2 * warp + par) * R;
        auto d1 = [&](int j, bool first) {
          if (elect_one())
            mma_tf32_ts(dst, tmem + L::cWQ + 8 * j, dadd(dS32, (j >> 2) * (R * 128) + (j & 3) * 32), id1, !first);
        };
        if constexpr (L::ND1 == 1) {
          issue_range<0, 16>(d1);
        } else {  // K steps 0-7, 8-15
          if (warp == 0) issue_range<0, 8>(d1);
          else issue_range<8, 16>(d1);
        }
        if (elect_one()) mma_commit(bar_d1);
        __syncwarp();
      }
      // (the factors of this chunk have landed: the prep waited for them before NB_W)
      if (quad < 2) {  // U = U~ - W S0^T (token t); U^ hi and lo (MN-major), U^T tf32
        wait(bar_d1, par);
        tc_fence_after();
        const float sc = gate[64 + t];
        if constexpr (L::NARROW) {
          // U^ rows first, then this warp's half of K^T U^ (the K steps of its own 32 tokens, so no
          // other warp's rows are needed), then U^T for P U while that half runs.
          float ut[32], dw[32];
          tmem_ld32(tmem + lane_base + L::cU + par * R, ut);
          tmem_ld32(tmem + lane_base + L::cD1 + par * R, dw);
          tmem_ld_wait();
          // U^ = sc U as bf16 hi + lo, both truncated (|error| < 2^-15 |U^|)
          __align__(16) uint32_t hp[16], lp[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float u0 = ut[i] - dw[i], u1 = ut[i + 1] - dw[i + 1];
            ut[i] = u0;
            ut[i + 1] = u1;
            const float h0 = u0 * sc, h1 = u1 * sc;
            const float t0 = __uint_as_float(__float_as_uint(h0) & 0xffff0000u);
            const float t1 = __uint_as_float(__float_as_uint(h1) & 0xffff0000u);
            hp[i / 2] = bf16x2_trunc(t0, t1);
            lp[i / 2] = bf16x2_trunc(h0 - t0, h1 - t1);
          }
#pragma unroll
          for (int i = 0; i < 32; i += 8) {  // N = 2R: hi in MN columns [0, R), lo in [R, 2R); K = 64 tokens
            *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(i, t, 64)) = *reinterpret_cast<const uint4*>(hp + i / 2);
            *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(R + i, t, 64)) = *reinterpret_cast<const uint4*>(lp + i / 2);
          }
          fence_async_smem();
          __syncwarp();
          {  // [K^T U^hi | K^T U^lo] over tokens [32 quad, 32 quad + 32): K steps 2 quad, 2 quad + 1
            const uint64_t dk = dadd(dKmn, kbuf(c) * 16384u + (uint32_t)quad * 4096u);
            const uint64_t du = dadd(dUHmn, (uint32_t)quad * 4096u);
            const uint32_t dst = tmem + L::cD2 + (uint32_t)quad * (2 * R);
            constexpr uint32_t id2 = idesc_bf16(128, 2 * R, true, true);
            auto d2 = [&](int j, bool first) {
              if (elect_one()) mma_bf16(dst, dadd(dk, j * 2048), dadd(du, j * 2048), id2, !first);
            };
            issue_range<0, 2>(d2);
            if (elect_one()) mma_commit(bar_d2);
            __syncwarp();
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) *reinterpret_cast<float*>(sm + L::UT + kf32(i, t, R)) = tf32r(ut[i]);
        } else {
#pragma unroll
          for (int hh = 0; hh < R / 32; ++hh) {  // 32 state rows at a time
            float ut[32], dw[32], x[32];
            tmem_ld32(tmem + lane_base + L::cU + par * R + 32 * hh, ut);
            tmem_ld32(tmem + lane_base + L::cD1 + par * R + 32 * hh, dw);
            if constexpr (L::ND1 == 2) tmem_ld32(tmem + lane_base + L::cD1 + (2 + par) * R + 32 * hh, x);
            tmem_ld_wait();
            if constexpr (L::ND1 == 2) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 w = __fadd2_rn(make_float2(dw[i], dw[i + 1]), make_float2(x[i], x[i + 1]));
                dw[i] = w.x;
                dw[i + 1] = w.y;
              }
            }
            // U^ = sc U as bf16 hi + lo, both truncated (|error| < 2^-15 |U^|)
            __align__(16) uint32_t hp[16], lp[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const int r = 32 * hh + i;
              const float u0 = ut[i] - dw[i], u1 = ut[i + 1] - dw[i + 1];
              *reinterpret_cast<float*>(sm + L::UT + kf32(r, t, R)) = tf32r(u0);
              *reinterpret_cast<float*>(sm + L::UT + kf32(r + 1, t, R)) = tf32r(u1);
              const float h0 = u0 * sc, h1 = u1 * sc;
              const float t0 = __uint_as_float(__float_as_uint(h0) & 0xffff0000u);
              const float t1 = __uint_as_float(__float_as_uint(h1) & 0xffff0000u);
              hp[i / 2] = bf16x2_trunc(t0, t1);
              lp[i / 2] = bf16x2_trunc(h0 - t0, h1 - t1);
            }
#pragma unroll
            for (int i = 0; i < 32; i += 8) {  // K = 128: hi in token rows 0-63, lo in 64-127
              const int r = 32 * hh + i;
              *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(r, t, 128)) = *reinterpret_cast<const uint4*>(hp + i / 2);
              *reinterpret_cast<uint4*>(sm + L::UH + mnbf16(r, 64 + t, 128)) = *reinterpret_cast<const uint4*>(lp + i / 2);
            }
          }
        }
      } else if (p.write_O && c > 0) {
        outputs(c - 1);
      }
      fence_async_smem();
      tc_fence_before();
      group_sync(1);
      // (64-row slices) K^T U^ (state) from warp 0; P U (outputs, P in rows 64-127) from warp 1
      if (!L::NARROW && warp == 0) {
        tc_fence_after();
        const uint64_t dk = dadd(dKmn, kbuf(c) * 16384u);
        // [K^T | K^T] [U^hi; U^lo]: K = 128
        constexpr uint32_t id2 = idesc_bf16(128, R, true, true);
        auto d2 = [&](int j, bool first) {
          if (elect_one()) mma_bf16(tmem + L::cD2, dadd(dk, (j & 3) * 2048), dadd(dUHmn, j * 2048), id2, !first);
        };
        issue_range<0, 8>(d2);
        if (elect_one()) mma_commit(bar_d2);
        __syncwarp();
      } else if ((warp & 1) == 1 && (warp >> 1) < L::NPU && p.write_O) {
        const uint32_t dst = tmem + L::cPU + (warp >> 1) * R;
        constexpr uint32_t idp = idesc_tf32(128, R);
        if constexpr (L::NARROW) {  // A = P from TMEM (lanes 64-127 of cMP)
          named_sync(NB_P, 96);
          tc_fence_after();
          auto pu = [&](int j, bool first) {
            if (elect_one())
              mma_tf32_ts(dst, tmem + L::cMP + 8 * j, dadd(dUT, (j >> 2) * (R * 128) + (j & 3) * 32), idp, !first);
          };
          issue_range<0, 8>(pu);
        } else {
          tc_fence_after();
          const uint64_t dp = dadd(dR2p, par * 18432);
          auto pu = [&](int j, bool first) {
            if (elect_one())
              mma_tf32(dst, dadd(dp, (j >> 2) * 8192 + (j & 3) * 32), dadd(dUT, (j >> 2) * (R * 128) + (j & 3) * 32),
                       idp, !first);
          };
          issue_range<0, 8>(pu);
        }
        if (elect_one()) mma_commit(bar_pu);
        __syncwarp();
      }
      if (p.write_O) gq_prev = gate[128 + t];  // output gate of this chunk (written out in the next)
      wait(bar_d2, par);
      tc_fence_after();
      {  // S <- gamma_C S + K^T U^ (M=128 layout: lane = d_k)
        const float gC = gate[63];
#pragma unroll
        for (int hh = 0; hh < R / 32; ++hh) {
          float d2[32], x[32], y[32], z[32];  // (32-row slices) [hi | lo] of both accumulators
          tmem_ld32(tmem + lane_base + L::cD2 + 32 * hh, d2);
          if constexpr (L::NARROW) {
            tmem_ld32(tmem + lane_base + L::cD2 + R, x);
            tmem_ld32(tmem + lane_base + L::cD2 + 2 * R, y);
            tmem_ld32(tmem + lane_base + L::cD2 + 3 * R, z);
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {  // packed pairs (same rounding as the scalar forms)
            const int r = 32 * hh + i;
            float2 d = make_float2(d2[i], d2[i + 1]);
            if constexpr (L::NARROW)
              d = __fadd2_rn(__fadd2_rn(d, make_float2(x[i], x[i + 1])),
                             __fadd2_rn(make_float2(y[i], y[i + 1]), make_float2(z[i], z[i + 1])));
            const float2 sn = __ffma2_rn(make_float2(gC, gC), make_float2(sreg[r], sreg[r + 1]), d);
            sreg[r] = sn.x;
            sreg[r + 1] = sn.y;
            *reinterpret_cast<float*>(sm + L::S32 + kf32(r, dcol, R)) = tf32r(sn.x);
            *reinterpret_cast<float*>(sm + L::S32 + kf32(r + 1, dcol, R)) = tf32r(sn.y);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_arrive(NB_S, 256);
    }
    if (p.write_O && nch > 0 && quad >= 2) outputs(nch - 1);
  } else {
    // ============================================================ prep warps
    const int t = 32 * (quad & 1) + lane;  // token of this thread's TMEM lane (rows of its quarter)
    for (int c = 0; c < nch; ++c) {
      const uint32_t par = c & 1;
      // (three K, two Q buffers) K and Q of chunk c+1, a chunk ahead: K goes to the buffer of
      // chunk c-2, Q to that of chunk c-1; their readers (W, K^T U^ of c-2; the Q rows of c-1)
      // finished before the chain ended chunk c-2, which the previous iteration waited for.
      // bar_kq[(c+1)&1] last completed for chunk c-1, also waited for: no phase overrun.
      if (L::EARLY_KQ && warp == 6 && elect_one() && c + 1 < nch) load_kq(c + 1);
      __syncwarp();
      wait(bar_kq + par, (c >> 1) & 1);
      wait(bar_r1, par);
      if constexpr (L::NARROW) {
        // Mb (hi | lo, bf16 pairs) into lanes 0-63 of cMP: U~ of the previous chunk has read them
        // (its completion was waited for below); P U may still read these lanes as rows nobody uses.
        if (quad < 2) {
#pragma unroll 1
          for (int a = 0; a < 2; ++a) {  // a = 0: hi (K 0-63), a = 1: lo (K 64-127)
            float v[32];  // column j holds K elements (2j, 2j + 1) as a bf16 pair
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::R1 + kRecMB + kbf16(t, 64 * a + 8 * ch, 64));
              v[4 * ch] = __uint_as_float(raw.x);
              v[4 * ch + 1] = __uint_as_float(raw.y);
              v[4 * ch + 2] = __uint_as_float(raw.z);
              v[4 * ch + 3] = __uint_as_float(raw.w);
            }
            tmem_st32(tmem + lane_base + L::cMP + 32 * a, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        group_sync(2);
      }
      if (warp == 4) {  // W = Mw K into the [W;Q] columns (M=128: rows 64-127 are replaced by Q below)
        if (c > 0) wait(bar_d1, (c - 1) & 1);  // the previous [W;Q] S0^T has read the [W;Q] columns
        tc_fence_after();
        constexpr uint32_t idW = idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (elect_one())
            mma_bf16(tmem + L::cWQ, dadd(dR1, kRecMW + j * 32), dadd(dKmn, kbuf(c) * 16384 + j * 2048), idW, j > 0);
        if (elect_one()) mma_commit(bar_w);
        __syncwarp();
      } else if (warp == 6) {  // U~ = [Mb_hi|Mb_lo][V;V] (M=128: rows 64-127 are not used)
        tc_fence_after();
        constexpr uint32_t idU = idesc_bf16(128, R, false, true);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (elect_one()) {
            if constexpr (L::NARROW)
              mma_bf16_ts(tmem + L::cU + par * R, tmem + L::cMP + 8 * j, dadd(dVT, (j & 3) * 2048), idU, j > 0);
            else
              mma_bf16(tmem + L::cU + par * R, dadd(dR1, kRecMB + (j >> 2) * 8192 + (j & 3) * 32),
                       dadd(dVT, (j & 3) * 2048), idU, j > 0);
          }
        }
        if (elect_one()) mma_commit(bar_u);
        __syncwarp();
      }
      wait(bar_w, par);
      wait(bar_u, par);
      tc_fence_after();
      group_sync(2);
      if (warp == 6 && elect_one() && c + 1 < nch) load_r1(c + 1);  // V and record part 1 are free
      __syncwarp();
      if (quad >= 2 && p.write_O) {  // Q rows (token 32*(quad-2) + lane): bf16, exact in fp32
        const int tq = 32 * (quad - 2) + lane;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {  // d_k columns [32 cc, 32 cc + 32)
          float v[32];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::QB + qbuf(c) * 16384 + kbf16(tq, cc * 32 + ch * 8, 64));
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[ch * 8 + 2 * e] = __uint_as_float(w[e] << 16);
              v[ch * 8 + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
          }
          tmem_st32(tmem + lane_base + L::cWQ + cc * 32, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      // Publish chunk c once the chain has finished chunk c-1 (it then finds this chunk's
      // operands ready and continues with a named-barrier round trip), and once record part 2
      // (factors and P) of chunk c has landed: the chain reads the factors without waiting.
      wait(bar_r2 + par, (c >> 1) & 1);
      if (c > 0) named_sync(NB_S, 256);
      named_arrive(NB_W, 256);

      if constexpr (L::NARROW) {
        // P of chunk c into lanes 64-127 of cMP (P U of chunk c-1 has completed: the chain
        // finished that chunk), then tell the P U issuers.
        if (quad >= 2 && p.write_O) {
          if (c > 0) wait(bar_pu, (c - 1) & 1);  // P U of chunk c-1 has read lanes 64-127 of cMP
          tc_fence_after();
          const unsigned char* P = sm + L::R2 + par * 18432 + (kRecP - kRecPart1);
#pragma unroll 1
          for (int a = 0; a < 2; ++a) {  // tokens s in [32 a, 32 a + 32)
            float v[32];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const float4 x = *reinterpret_cast<const float4*>(P + kf32(t, 32 * a + 4 * ch, 64));
              v[4 * ch] = x.x;
              v[4 * ch + 1] = x.y;
              v[4 * ch + 2] = x.z;
              v[4 * ch + 3] = x.w;
            }
            tmem_st32(tmem + lane_base + L::cMP + 32 * a, v);
          }
          tmem_st_wait();
          tc_fence_before();
          named_arrive(NB_P, 96);
        }
      }
      if (warp == 6 && elect_one() && c + 1 < nch) {
        // (two K, one Q buffer) K of chunk c-1 and the Q staging buffer have no readers left
        if (!L::EARLY_KQ) load_kq(c + 1);
        if (c >= 1) load_r2(c + 1);  // P and factors of chunk c-1 are no longer read
      }
      __syncwarp();
    }
    if (nch > 0) named_sync(NB_S, 256);  // the chain's arrival for its last chunk
  }

  __syncthreads();
  if (flags[0]) {
    if (tid == 0) atomicExch(p.status, GDN_ERR_TIMEOUT);
  } else if (chain) {
#pragma unroll
    for (int c = 0; c < R; ++c) p.S_out[sbase + (size_t)(row0 + c) * DK + dcol] = sreg[c];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
}  // namespace

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

// 2D bf16 view [rows][cols] (cols contiguous), boxes of 64 columns x box_rows rows, 128-byte
// swizzle, zero fill out of range.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_f32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int R>
cudaError_t launch_scan(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const ScanParams& sp,
                        bool overlap_prep, cudaStream_t stream) {
  using L = ScanLay<R>;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::ALLOC);
  if (e != cudaSuccess) return e;
  // With overlap_prep the scan is a programmatic dependent of the prep kernel just before it on
  // the stream: its CTAs launch while the last prep CTAs run, set up and fetch the first K, Q
  // tiles, then wait for the prep grid before reading the records.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(DV / R, sp.h_v, sp.n_seqs);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap_prep ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_scan_kernel<R>, mq, mk, mv, sp);
}

}  // namespace

int replay_tc_rows(int n_seqs, int h_v) {
  // 4 slices of 32 state rows per (tail, v-head) while those fit on the GPU at once (latency);
  // 2 slices of 64 rows when there are more (throughput: the MMAs of a chunk take about as long
  // at N = 64 as at N = 32, so a 64-row CTA does twice the work in a little more time).
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  return (long long)n_seqs * h_v * (DV / 32) > sms ? 64 : 32;
}

bool replay_tc_supported(const SimtParams& p) {
  return p.d_k == DK && p.d_v == DV && p.total_tokens > 0 && p.n_seqs > 0 && !p.augmented;
}

namespace {
// Records of all chunks, then (several tails) the tail order.
size_t records_bytes(int n_seqs, int total_tokens, int h_v) {
  // chunks of all tails <= ceil(total / 64) + one partial chunk per tail
  const size_t chunks = (size_t)(total_tokens + C - 1) / C + (size_t)n_seqs;
  return (chunks * (size_t)h_v * kRecBytes + 255) / 256 * 256;
}

// Varlen work order: the tails ranked by length, longest first (ties by index), order[rank] =
// tail.  The scan's grid walks the tails in this order, so the longest replays start in the
// first wave and the last wave holds short ones (longest-processing-time-first list
// scheduling: the grid's makespan is then bounded by the average load plus a short tail
// rather than plus the longest one).  One thread per tail counts the tails ahead of it.
__global__ void tail_order_kernel(const int32_t* __restrict__ cu, int n, int32_t* __restrict__ order) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long li = (long long)cu[i + 1] - cu[i];
  int rank = 0;
  for (int j = 0; j < n; ++j) {
    const long long lj = (long long)cu[j + 1] - cu[j];
    rank += (lj > li) || (lj == li && j < i);
  }
  order[rank] = i;
}
}  // namespace

size_t replay_tc_workspace_bytes(int n_seqs, int total_tokens, int h_v) {
  return records_bytes(n_seqs, total_tokens, h_v) + (n_seqs > 1 ? (size_t)n_seqs * sizeof(int32_t) : 0);
}

cudaError_t launch_replay_tc(const SimtParams& p, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (workspace_bytes < replay_tc_workspace_bytes(p.n_seqs, p.total_tokens, p.h_v)) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  const void* qsrc = p.write_O ? p.q : p.k;  // q unused without outputs: any valid tile source
  if (!make_map(&mq, qsrc, p.total_tokens, (uint64_t)p.h_k * DK, 64) ||
      !make_map(&mk, p.k, p.total_tokens, (uint64_t)p.h_k * DK, 64) ||
      !make_map(&mv, p.v, p.total_tokens, (uint64_t)p.h_v * DV, 64))
    return cudaErrorInvalidValue;
  unsigned char* rec = static_cast<unsigned char*>(workspace);
  int32_t* order = nullptr;
  if (p.n_seqs > 1) {  // several tails: longest first
    order = reinterpret_cast<int32_t*>(rec + records_bytes(p.n_seqs, p.total_tokens, p.h_v));
    tail_order_kernel<<<(p.n_seqs + 255) / 256, 256, 0, stream>>>(p.cu, p.n_seqs, order);
    const cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
  }

  PrepParams pp;
  pp.g = p.g; pp.beta = p.beta; pp.cu = p.cu; pp.rec = rec; pp.status = p.status;
  pp.n_seqs = p.n_seqs; pp.total_tokens = p.total_tokens; pp.h_k = p.h_k; pp.h_v = p.h_v; pp.l2norm = p.l2norm;
  pp.write_O = p.write_O; pp.scale = p.scale; pp.scalar_decay = p.scalar_decay;
  // State-only calls with 32-row slices take the operator-form scan, which reads Z instead of Mw.
  const bool state_form = !p.write_O && replay_tc_rows(p.n_seqs, p.h_v) == 32;
  pp.zform = state_form ? 1 : 0;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PrepLay::ALLOC);
  if (e != cudaSuccess) return e;
  const long long items_ub = ((long long)(p.total_tokens + C - 1) / C + p.n_seqs) * p.h_k;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  const int grid = (int)std::min<long long>(items_ub, 2LL * sms);  // two CTAs per SM
  chunk_prep_kernel<<<grid, NT, PrepLay::ALLOC, stream>>>(mq, mk, pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bool overlap = true;  // a stage event between the kernels asks for them to run one after the other
  if (void* ev = take_stage_event()) {
    overlap = false;
    e = cudaEventRecord(static_cast<cudaEvent_t>(ev), stream);
    if (e != cudaSuccess) return e;
  }

  if (state_form) {
    StateParams st;
    st.cu = p.cu; st.order = order; st.S0 = p.S0; st.rec = rec; st.S_out = p.S_out; st.status = p.status;
    st.n_seqs = p.n_seqs; st.total_tokens = p.total_tokens; st.h_k = p.h_k; st.h_v = p.h_v;
    return launch_state_tc(mk, mv, st, overlap, stream);
  }
  ScanParams sp;
  sp.cu = p.cu; sp.order = order; sp.S0 = p.S0; sp.rec = rec; sp.O = static_cast<__nv_bfloat16*>(p.O); sp.S_out = p.S_out;
  sp.status = p.status; sp.n_seqs = p.n_seqs; sp.total_tokens = p.total_tokens; sp.h_k = p.h_k; sp.h_v = p.h_v;
  sp.write_O = p.write_O;
  return replay_tc_rows(p.n_seqs, p.h_v) == 64 ? launch_scan<64>(mq, mk, mv, sp, overlap, stream)
                                                : launch_scan<32>(mq, mk, mv, sp, overlap, stream);
}

}  // namespace gdn

// ---------------------------------------------------------------------------------------------
// Allocation-free replay: the same prep + scan kernels, with their scratch in a fixed static
// device array instead of the stream-ordered pool.
// ---------------------------------------------------------------------------------------------
namespace gdn {
namespace {

// 96 MiB on every GPU that loads the library, held until process exit.  Enough for the
// records of one 3277-token tail at 32 v-heads ((52 + 1) chunks x 32 heads x 41984 B = 67.9 MiB).
constexpr size_t kStaticScratchBytes = size_t(96) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  In host code the symbol itself is
// only a host-side stand-in, so the address is looked up on every call with the device current
// (no cached pointer can outlive a device reset).
int static_scratch_address(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
  if (e != cudaSuccess || !ptr) return report_error(GDN_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
  *out = ptr;
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
                          "gdn_replay_noalloc: the problem needs more scratch than the 96 MiB static array "
                          "(gdn_workspace_bytes gives the amount); use gdn_replay");
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
