// Tensor-core (tcgen05 + TMEM + TMA) state-only scan of the fp32 path, d_k = d_v = 128: the scan
// pass of gdn_chunk_operator (augmented state) at fp32 accuracy.
//
// Method: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix Caching for Hybrid
// LLMs", section 2 Eq. (1), chunk by chunk (C = 64 tokens), in the form the fp32 path's header
// derives: with the chunk's record (M = (I + A)^{-1}, gamma_t, exp(G_C - G_t), beta_t, the key
// norm factors rk_t) and the entering state X (rows r, columns k):
//   Y  = X K^T diag(rk)                          (row r, token t)
//   R  = (V^T - Y diag(gamma)) diag(beta)        (no Y term in the scalar-decay family)
//   U  = R M^T
//   X' = gamma_C X + U diag(rk exp(G_C - G_t)) K
// "LinearKV: One Cached State Suffices for Position-Independent Caching in Hybrid LLMs",
// composition passage: the operator's transition part rides along as d_k extra state rows,
// seeded with the identity and fed zero values (X = [S; P], P = T_C^T after the chunk).
//
// One CTA owns 128 state rows of one (sequence, v-head): TMEM lane r = state row r, and every
// product keeps that orientation, so each result is read back by the thread that owns its row.
// Each of the three contractions runs in split tf32 (three tensor-core products: hi*hi, hi*lo,
// lo*hi; the tensor core reads an fp32 operand as tf32 by dropping its low 13 mantissa bits, so
// an fp32 value in memory serves as its own hi part and lo = x - hi is exact):
//   D1 = X [K; K_lo]^T       A = X (TMEM), B = K tile, 128 rows: tokens, then their lo parts
//        + X_lo K^T          A = X - X_hi (TMEM), B = the first 64 rows
//   D2 = R [M; M_lo]^T + R_lo M^T                  (A in TMEM, B = M tile of 128 rows)
//   D3 = U^ K^T + U^ K_lo^T + U^_lo K^T            (B = K transposed by the threads: a tf32
//                                                   operand must be K-major)
// and the epilogues add the hi*lo halves in fp32.  The state stays in fp32 registers.
// With bf16 inputs the keys and values are exact in tf32, so the key lo parts vanish: D1 is
// X K^T + X_lo K^T (N = 64) and D3 U^ K^T + U^_lo K^T; the keys arrive by 16-byte loads into
// registers during the previous piece's state update instead of by TMA.
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace tcp;

constexpr int C = kChunk;  // 64 tokens
constexpr int D = 128;     // d_k = d_v; state rows per CTA
constexpr int NT = 256;    // 8 warps: two per TMEM sub-partition

struct COLay {
  static constexpr uint32_t KT = 0;            // 2 buffers of [K; K_lo]: fp32 K-major, 4 atoms x 128 rows x 128 B
  static constexpr uint32_t KTBUF = 65536;
  static constexpr uint32_t KTT = 2 * KTBUF;   // K^T, then K_lo^T: K-major [k][t], 2 atoms x 128 rows x 128 B each
  static constexpr uint32_t MT = KTT + 65536;  // [M; M_lo]: K-major [t][s], 2 atoms x 128 rows x 128 B
  static constexpr uint32_t FAC = MT + 32768;  // per token: gamma, exp(G_C - G_t), beta, rk (4 x 64 floats)
  static constexpr uint32_t BARS = FAC + 1024;
  static constexpr uint32_t TOTAL = BARS + 64;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
  // TMEM: X (then D3), X_lo, D1 (then R | R_lo), D2 (then U^ | U^_lo)
  static constexpr uint32_t cX = 0, cXL = 128, cD1 = 256, cD2 = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(ALLOC <= 232448, "shared memory");
};

struct COParams {
  const void* k;  // keys (bf16 inputs; fp32 keys arrive by TMA)
  const void* v;
  const float* S0;
  const int32_t* cu;
  const float* rec;
  float* S_out;
  float* T_out;
  int* status;
  int n_seqs, total_tokens, h_k, h_v, augmented, scalar_decay;
};

__device__ __forceinline__ float tf32_lo(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ __forceinline__ float ld_val(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_val(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }

template <bool BF16>
__global__ void __launch_bounds__(NT, 1) chunkop_tc_kernel(const __grid_constant__ CUtensorMap map_k, const COParams p) {
  using Tin = typename std::conditional<BF16, __nv_bfloat16, float>::type;
  using L = COLay;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* fGam = reinterpret_cast<float*>(sm + L::FAC);
  float* fWend = fGam + 64;
  float* fBeta = fGam + 128;
  float* fRk = fGam + 192;
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_k = bar_mma + 1;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::BARS + 24);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, hf = warp >> 2;
  const int slice = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int r = 32 * quad + lane;  // state row in the slice = TMEM lane
  const int rg = slice * D + r;    // row of the (augmented) state
  const int hk = h / (p.h_v / p.h_k);

  // A malformed range (see chunk_info) is skipped and reported; `first` is the global index of
  // this sequence's first chunk in the records.  (chunk_info's scratch: the factor area.)
  int first = 0;
  if (p.cu) {
    const ChunkInfo ci = chunk_info(p.cu, p.n_seqs, p.total_tokens, seq, -1, reinterpret_cast<int*>(sm + L::FAC));
    if (!ci.valid) {
      if (tid == 0) atomicExch(p.status, GDN_ERR_SHAPE);
      return;
    }
    first = ci.first;
  }
  __syncthreads();  // chunk_info's scratch (the factor area) is free again
  const int t_begin = p.cu ? p.cu[seq] : 0;
  const int t_end = p.cu ? p.cu[seq + 1] : p.total_tokens;
  const int n_chunks = (t_end - t_begin + C - 1) / C;

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  auto issue_k = [&](int c) {  // one thread: chunk c's raw keys into rows 0-63 of buffer c & 1
    const int b = c & 1;
    mbar_arrive_expect_tx(&bar_k[b], 4 * 8192);
#pragma unroll
    for (int a = 0; a < 4; ++a)
      tma_load_2d(sm + L::KT + b * L::KTBUF + a * 16384, &map_k, &bar_k[b], hk * D + 32 * a, t_begin + c * C);
  };
  if (tid == 0) {
    mbar_init(bar_mma, 1);
    mbar_init(&bar_k[0], 1);
    mbar_init(&bar_k[1], 1);
    mbar_fence_init();
    if constexpr (!BF16) {
      tma_prefetch_desc(&map_k);
      if (n_chunks > 0) issue_k(0);
    }
  }
  // entering state of this thread's row, columns [64 hf, 64 hf + 64): S0 rows, or identity rows
  float x[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const int k = 64 * hf + i;
    float s = 0.f;
    if (rg < D) {
      if (p.S0) s = p.S0[(((size_t)seq * p.h_v + h) * D + rg) * D + k];
    } else {
      s = (k == rg - D) ? 1.f : 0.f;
    }
    x[i] = s;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  auto store_x = [&]() {  // X and X - X_hi into TMEM (this thread's lane and columns)
    float w[32];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      tmem_st32(tmem + lane_base + L::cX + 64 * hf + 32 * c2, *reinterpret_cast<const float(*)[32]>(x + 32 * c2));
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = tf32_lo(x[32 * c2 + i]);
      tmem_st32(tmem + lane_base + L::cXL + 64 * hf + 32 * c2, w);
    }
  };
  store_x();

  int timed_out = 0;
  uint32_t mph = 0;  // phase of bar_mma
  int k_issued = (!BF16 && n_chunks > 0) ? 0 : -1, k_waited = -1;  // key copies (fp32 keys only)
  auto wait_mma = [&]() {
    if (!mbar_wait(bar_mma, mph & 1u, kWaitNs)) timed_out = 1;
    ++mph;
    tc_fence_after();
  };
  // chunk c's M (and its lo part) into the M tile; this thread's one of the 256 factor floats
  // (gamma, exp(G_C - G_t), beta, rk) is returned, for the factor table once its readers are done
  auto load_rec = [&](int c) {
    const float* Rc = p.rec + ((size_t)(first + c) * p.h_v + h) * REC_FLOATS;
    float4 mv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) mv[j] = *reinterpret_cast<const float4*>(Rc + REC_M + (tid + j * NT) * 4);
    const float fac = Rc[REC_GAM + tid];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // M (row t, columns s4..s4+3) and its lo part
      const int i4 = tid + j * NT, t = i4 >> 4, s4 = (i4 & 15) * 4;
      const float4 m = mv[j];
      *reinterpret_cast<float4*>(sm + L::MT + kf32(t, s4, 128)) = m;
      *reinterpret_cast<float4*>(sm + L::MT + kf32(64 + t, s4, 128)) =
          make_float4(tf32_lo(m.x), tf32_lo(m.y), tf32_lo(m.z), tf32_lo(m.w));
    }
    return fac;
  };
  float fac_next = n_chunks > 0 ? load_rec(0) : 0.f;
  // bf16 keys of piece c: warp w, step j covers the 8 columns 8 ((w + 8 j) & 15) + [0, 8) of token
  // lane + 32 ((w + 8 j) >> 4) (zero past the piece's end)
  uint4 kq[4];
  auto load_k16 = [&](int c) {
    const int t0c = t_begin + c * C, nc = min(C, t_end - t0c);
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(p.k);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int combo = warp + 8 * j, oct = combo & 15, t = lane + 32 * (combo >> 4);
      kq[j] = t < nc ? *reinterpret_cast<const uint4*>(kb + ((size_t)(t0c + t) * p.h_k + hk) * D + 8 * oct)
                     : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if constexpr (BF16) {
    if (n_chunks > 0) load_k16(0);
  }
  // values of piece c for this thread's row and tokens [32 hf, +32) (transition rows: zero)
  auto load_v = [&](int c, float (&out)[32]) {
    const int t0c = t_begin + c * C, nc = min(C, t_end - t0c);
    if (slice == 0) {
      const Tin* vp = static_cast<const Tin*>(p.v) + ((size_t)(t0c + 32 * hf) * p.h_v + h) * D + rg;
      const size_t vs = (size_t)p.h_v * D;
      const int nv = nc - 32 * hf;  // tokens of this thread's half that exist
#pragma unroll
      for (int i = 0; i < 32; ++i) out[i] = i < nv ? ld_val(vp, i * vs) : 0.f;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) out[i] = 0.f;
    }
  };
  // fp32 inputs: the next piece's values are loaded during the current state update (the loads
  // then wait on memory while the threads would wait on the MMAs anyway)
  float vnext[32];
  if constexpr (!BF16) {
    if (n_chunks > 0) load_v(0, vnext);
  }
  const uint64_t dKTT = sdesc_sw128(smem_u32(sm + L::KTT), 16, 1024);
  const uint64_t dMT = sdesc_sw128(smem_u32(sm + L::MT), 16, 1024);
  constexpr uint32_t id128 = idesc_tf32(128, 128);
  constexpr uint32_t id64 = idesc_tf32(128, 64);

  for (int c = 0; c < n_chunks; ++c) {
    const int t0 = t_begin + c * C, n = min(C, t_end - t0);
    const int b = BF16 ? 0 : (c & 1);  // (bf16 keys: one buffer, filled by the threads)
    unsigned char* kt = sm + L::KT + b * L::KTBUF;
    // fp32 keys: the next chunk's raw keys into the other buffer (its last readers, chunk c - 1's
    // D1 and transposition, finished before that chunk's state update)
    if (tid == 0 && c + 1 < n_chunks) {
      if constexpr (!BF16) {
        issue_k(c + 1);
        k_issued = c + 1;
      }
      // and its M and factors into L2 (read while this chunk's state update runs)
      const float* Rn = p.rec + ((size_t)(first + c + 1) * p.h_v + h) * REC_FLOATS;
      bulk_prefetch_l2(Rn + REC_M, 4096 * 4);
      bulk_prefetch_l2(Rn + REC_GAM, 256 * 4);
    }
    // this chunk's factors (loaded during the previous state update; their readers are done)
    fGam[tid] = fac_next;
    // this chunk's values (row r, tokens [32 hf, +32)): fp32 loaded during the previous state
    // update; bf16 loaded here, in flight while the keys are transposed
    float vv[32];
    if constexpr (BF16) {
      load_v(c, vv);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) vv[i] = vnext[i];
    }
    if constexpr (BF16) {
      // bf16 keys from registers: fp32 rows 0-63 of the key tile and K^T (token lane in each
      // K^T store: whole 128-byte rows)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int combo = warp + 8 * j, oct = combo & 15, t = lane + 32 * (combo >> 4);
        const uint32_t w[4] = {kq[j].x, kq[j].y, kq[j].z, kq[j].w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = __uint_as_float(w[e] << 16);
          f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
        *reinterpret_cast<float4*>(kt + kf32(t, 8 * oct, 128)) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(kt + kf32(t, 8 * oct + 4, 128)) = make_float4(f[4], f[5], f[6], f[7]);
#pragma unroll
        for (int e = 0; e < 8; ++e) *reinterpret_cast<float*>(sm + L::KTT + kf32(8 * oct + e, t, 128)) = f[e];
      }
    } else {
      if (!mbar_wait(&bar_k[b], (uint32_t)((c >> 1) & 1), kWaitNs)) timed_out = 1;
      k_waited = c;
      // keys: rows past the chunk's end (the next sequence's tokens, or the fill) cleared; lo parts
      // into rows 64-127; K^T and K_lo^T (row k, token t) for the state update.  Warp w, step i:
      // columns 4 (w + 8 i) + [0, 4) of tokens lane and lane + 32 (a warp's K^T stores fill whole
      // 128-byte rows; every access of the loop takes the fewest shared-memory wavefronts).
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kc = warp + 8 * i;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int t = lane + 32 * hh;
          float4* src = reinterpret_cast<float4*>(kt + kf32(t, 4 * kc, 128));
          float4 kv = *src;
          if (t >= n) {
            kv = make_float4(0.f, 0.f, 0.f, 0.f);
            *src = kv;
          }
          const float4 lo = make_float4(tf32_lo(kv.x), tf32_lo(kv.y), tf32_lo(kv.z), tf32_lo(kv.w));
          *reinterpret_cast<float4*>(kt + kf32(64 + t, 4 * kc, 128)) = lo;
          const float kr[4] = {kv.x, kv.y, kv.z, kv.w}, kl[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            *reinterpret_cast<float*>(sm + L::KTT + kf32(4 * kc + e, t, 128)) = kr[e];
            *reinterpret_cast<float*>(sm + L::KTT + 32768 + kf32(4 * kc + e, t, 128)) = kl[e];
          }
        }
      }
    }
    tmem_st_wait();  // X, X_lo (previous state update)
    fence_async_smem();
    tc_fence_before();
    if (__syncthreads_or(timed_out)) break;
    tc_fence_after();
    // D1 = X [K; K_lo]^T + X_lo K^T
    if (tid == 0) {
      const uint64_t dK = sdesc_sw128(smem_u32(kt), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint64_t bk = dK + (uint64_t)((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4);
        mma_tf32_ts(tmem + L::cD1, tmem + L::cX + 8 * kk, bk, BF16 ? id64 : id128, kk > 0);
        mma_tf32_ts(tmem + L::cD1, tmem + L::cXL + 8 * kk, bk, id64, 1);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_mma();
    // R (row r, tokens [32 hf, +32)) = beta (v - gamma rk (X K^T)), written over D1
    {
      float a[32], bb[32];
      tmem_ld32(tmem + lane_base + L::cD1 + 32 * hf, a);
      if constexpr (!BF16) tmem_ld32(tmem + lane_base + L::cD1 + 64 + 32 * hf, bb);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = 32 * hf + i;
        const float y = (BF16 ? a[i] : a[i] + bb[i]) * fRk[t];
        a[i] = fBeta[t] * (p.scalar_decay ? vv[i] : fmaf(-fGam[t], y, vv[i]));
        bb[i] = tf32_lo(a[i]);
      }
      tmem_st32(tmem + lane_base + L::cD1 + 32 * hf, a);
      tmem_st32(tmem + lane_base + L::cD1 + 64 + 32 * hf, bb);
      tmem_st_wait();
    }
    tc_fence_before();
    if (__syncthreads_or(timed_out)) break;
    tc_fence_after();
    // D2 = R [M; M_lo]^T + R_lo M^T
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t bm = dMT + (uint64_t)((((ks >> 2) * 16384) + (ks & 3) * 32) >> 4);
        mma_tf32_ts(tmem + L::cD2, tmem + L::cD1 + 8 * ks, bm, id128, ks > 0);
        mma_tf32_ts(tmem + L::cD2, tmem + L::cD1 + 64 + 8 * ks, bm, id64, 1);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_mma();
    // U^ = U diag(rk exp(G_C - G_t)), written over D2
    {
      float a[32], bb[32];
      tmem_ld32(tmem + lane_base + L::cD2 + 32 * hf, a);
      tmem_ld32(tmem + lane_base + L::cD2 + 64 + 32 * hf, bb);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = 32 * hf + i;
        a[i] = (a[i] + bb[i]) * (fWend[t] * fRk[t]);
        bb[i] = tf32_lo(a[i]);
      }
      tmem_st32(tmem + lane_base + L::cD2 + 32 * hf, a);
      tmem_st32(tmem + lane_base + L::cD2 + 64 + 32 * hf, bb);
      tmem_st_wait();
    }
    tc_fence_before();
    if (__syncthreads_or(timed_out)) break;
    tc_fence_after();
    // D3 = U^ K^T + U^ K_lo^T + U^_lo K^T, over X's columns (X was read only by D1)
    if (tid == 0) {
#pragma unroll
      for (int ts = 0; ts < 8; ++ts) {
        const uint32_t off = (((ts >> 2) * 16384) + (ts & 3) * 32) >> 4;
        mma_tf32_ts(tmem + L::cX, tmem + L::cD2 + 8 * ts, dKTT + off, id128, ts > 0);
        if constexpr (!BF16) mma_tf32_ts(tmem + L::cX, tmem + L::cD2 + 8 * ts, dKTT + (32768 >> 4) + off, id128, 1);
        mma_tf32_ts(tmem + L::cX, tmem + L::cD2 + 64 + 8 * ts, dKTT + off, id128, 1);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    // while the state update runs: the next chunk's M into the M tile (its reader, D2, is done)
    if (c + 1 < n_chunks) {
      fac_next = load_rec(c + 1);
      if constexpr (BF16) load_k16(c + 1);  // (into registers; they fill the key tile at the next piece's top)
      else load_v(c + 1, vnext);
    }
    wait_mma();
    // X <- gamma_C X + D3, and X, X_lo into TMEM for the next chunk
    {
      const float gC = fGam[C - 1];
      float d3[32];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        tmem_ld32(tmem + lane_base + L::cX + 64 * hf + 32 * c2, d3);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[32 * c2 + i] = fmaf(gC, x[32 * c2 + i], d3[i]);
      }
      store_x();
    }
    tc_fence_before();
    if (__syncthreads_or(timed_out)) break;  // also: every read of this chunk's M and factors is done
    tc_fence_after();
  }

  tc_fence_before();
  if (__syncthreads_or(timed_out)) {
    // A wait gave up: let the key copy in flight land and the MMAs finish (each wait bounded),
    // then report.  The results are unspecified.
    if (tid == 0) {
      if (k_issued > k_waited) mbar_wait(&bar_k[k_issued & 1], (uint32_t)((k_issued >> 1) & 1), kWaitNs);
      if (mph > 0) mbar_wait(bar_mma, (mph - 1) & 1u, kWaitNs);
      atomicExch(p.status, GDN_ERR_TIMEOUT);
    }
    __syncthreads();
  } else {
    // final state: value rows to S_out, transition rows (P = T_C^T) to T_out transposed
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const int k = 64 * hf + i;
      if (rg < D) {
        p.S_out[(((size_t)seq * p.h_v + h) * D + rg) * D + k] = x[i];
      } else {
        p.T_out[(((size_t)seq * p.h_v + h) * D + k) * D + (rg - D)] = x[i];
      }
    }
  }
  tmem_st_wait();  // the last state stores into TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace

bool chunkop_tc_supported(const SimtParams& p, int bf16) {
  (void)bf16;
  return !p.write_O && p.rec && p.d_k == D && p.d_v == D && p.total_tokens > 0;
}

cudaError_t launch_chunkop_tc(const SimtParams& sp, int bf16, cudaStream_t stream) {
  CUtensorMap map{};  // (bf16 keys are loaded by the threads: no map)
  if (!bf16 && !make_map_f32(&map, sp.k, (uint64_t)sp.total_tokens, (uint64_t)sp.h_k * D, kChunk))
    return cudaErrorInvalidValue;
  COParams p{};
  p.k = sp.k;
  p.v = sp.v;
  p.S0 = sp.S0;
  p.cu = sp.cu;
  p.rec = reinterpret_cast<const float*>(sp.rec);
  p.S_out = sp.S_out;
  p.T_out = sp.T_out;
  p.status = sp.status;
  p.n_seqs = sp.n_seqs;
  p.total_tokens = sp.total_tokens;
  p.h_k = sp.h_k;
  p.h_v = sp.h_v;
  p.augmented = sp.augmented;
  p.scalar_decay = sp.scalar_decay;
  const dim3 grid(sp.augmented ? 2 : 1, sp.h_v, sp.n_seqs);
  auto kern = bf16 ? chunkop_tc_kernel<true> : chunkop_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)COLay::ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<grid, NT, COLay::ALLOC, stream>>>(map, p);
  return cudaGetLastError();
}

}  // namespace gdn
