// fp32 chunked scan: the precise path of gdn_replay (fp32 inputs, other head
// sizes, or bf16 inputs with GDN_PRECISE) and the whole of gdn_chunk_operator.
// fp32 data throughout; the contractions run on warp-level tensor cores
// (mma.sync) in split tf32, about 21 significant bits.
//
// Method: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix
// Caching for Hybrid LLMs", section 2 Eq. (1) and section 3 Eq. (2), run
// chunk by chunk.  Within a chunk of C = 64 tokens with inclusive gate sums
// G_t (gamma_t = exp(G_t)) and entering state S0, unrolling Eq. (1) gives
//     S_t = gamma_t S0 + sum_{s<=t} exp(G_t - G_s) u_s k_s^T,
// where the corrected values u_s solve the unit lower-triangular system
//     (I + A) U = diag(beta) (V - diag(gamma) K S0^T),
//     A_ts = beta_t exp(G_t - G_s) k_t.k_s   (s < t).
// Hence, with M = (I + A)^{-1}:
//     U      = M diag(beta) (V - diag(gamma) K S0^T)
//     S_end  = gamma_C S0 + U^T diag(exp(G_C - G_s)) K
//     O      = diag(gamma) Q S0^T + (L o Q K^T) U,   L_ts = exp(G_t - G_s), s <= t.
// Only S is carried from chunk to chunk, in fp32.
//
// Chunk-operator mode ("LinearKV: One Cached State Suffices for
// Position-Independent Caching in Hybrid LLMs", composition passage): the
// state gains d_k extra rows P, seeded with the identity and fed zero values.
// Rows evolve independently, so after the chunk P = T_1 ... T_n
// (right-multiplied form) = T_C^T, written transposed as T_C.
//
// One CTA owns a 32-row slice of one (sequence, v-head) state and walks its
// chunks.  gdn_replay and gdn_chunk_operator run two passes: the chunk-shared
// quantities (norms, gates, M, P) once per (chunk, v-head) into a record, then
// the slices read them; the allocation-free replay computes them in every
// slice (one pass, no scratch).  Partial last chunks are padded with tokens that have k = 0,
// beta = 0, g = 0: identity transitions whose outputs are not stored.
#include <cuda_bf16.h>

#include <cstddef>

#include "gdn_internal.cuh"
#include "tc_common.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;
constexpr int RS = 32;                // state rows per CTA
// Row strides (floats) chosen for the m16n8k8 fragments: rows 4 (K/Q/S, 64x64) or 8 (V/R/U)
// banks apart, so the eight rows and four columns a fragment load touches hit distinct banks.
constexpr int KST = kMaxHead + 4;     // K/Q/S tiles
constexpr int VST = RS + 8;           // V/R/U/X tiles
constexpr int GST = C + 4;            // the 64x64 tiles
constexpr int NT = 256;

struct Smem {
  float K[C * KST];
  float K2[C * KST];   // second key buffer: the next chunk's keys arrive while this one is used
  float Q[C * KST];
  float S[RS * KST];
  float V[C * VST];    // values, then R, then U
  float A[C * GST];    // strictly lower A
  float P[C * GST];    // (L o Q K^T), inclusive lower
  float M[C * GST];    // (I + A)^{-1}
  float X[C * VST];    // K S0^T
  float G[C];          // inclusive gate sums
  float gam[C];        // exp(G_t)
  float wend[C];       // exp(G_last - G_t)
  float beta[C];
  float rk[C];         // key norm factors of the record path (gam, wend, beta, rk are contiguous)
  int scratch[20];
};

// 16-byte asynchronous copy global -> shared (zero-filled when !valid; src must still be mapped).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// The C fragments of a warp's two 16 x 8 tiles (rows m0.., columns n0 + [0, 16)) into a
// row-major tile with row stride ld.
__device__ __forceinline__ void store_tile(float* T, int ld, const float (&acc)[2][4], int m0, int n0, int lane) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c = n0 + 8 * j + 2 * q;
    T[(m0 + g) * ld + c] = acc[j][0];
    T[(m0 + g) * ld + c + 1] = acc[j][1];
    T[(m0 + g + 8) * ld + c] = acc[j][2];
    T[(m0 + g + 8) * ld + c + 1] = acc[j][3];
  }
}

__device__ __forceinline__ float ld_in(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_out(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------------------------
// Two-pass mode: the chunk-shared quantities, once per (chunk, v-head), in the fp32 record
// layout of gdn_internal.cuh (REC_*).

struct PrepSmem {
  float K[C * KST];
  float A[2][C * tcp::MST];  // per v-head slot
  float M[2][C * tcp::MST];
  float G[2][C], beta[2][C], rk[C], rq[C];
  int scratch[20];
  float Q[C * KST];  // last: not allocated when no outputs are wanted
};
constexpr size_t kPrepSmemNoQ = offsetof(PrepSmem, Q);

// One CTA per (global chunk, key head, pair of its v-heads): load and normalise the chunk's keys
// (and queries) and form the Gram matrices once; then per v-head slot the gates, A and P, and
// M = (I + A)^{-1} (one warpgroup per slot); write the records.
template <typename Tin>
__global__ void __launch_bounds__(NT) simt_chunk_prep_kernel(SimtParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int gc = blockIdx.x;
  const int G_ = p.h_v / p.h_k, npairs = (G_ + 1) / 2;
  const int hk = blockIdx.y / npairs, pair = blockIdx.y % npairs;
  const int h0 = hk * G_ + 2 * pair, nslots = min(2, G_ - 2 * pair);  // v-heads h0, h0 + 1
  const int DK = p.d_k;
  int t0, n;
  if (p.cu) {
    const tcp::ChunkInfo ci = tcp::chunk_info(p.cu, p.n_seqs, p.total_tokens, -1, gc, sm.scratch);
    if (gc >= ci.total || ci.gc_seq < 0) return;
    t0 = p.cu[ci.gc_seq] + ci.gc_idx * C;
    n = min(C, p.cu[ci.gc_seq + 1] - t0);
  } else {
    if (gc >= tcp::chunks_of(p.total_tokens)) return;
    t0 = gc * C;
    n = min(C, p.total_tokens - t0);
  }
  const Tin* __restrict__ q = static_cast<const Tin*>(p.q);
  const Tin* __restrict__ k = static_cast<const Tin*>(p.k);
  auto rec_of = [&](int slot) { return reinterpret_cast<float*>(p.rec) + ((size_t)gc * p.h_v + h0 + slot) * REC_FLOATS; };

  bool loaded = false;
  if constexpr (sizeof(Tin) == 4) {
    if (DK == kMaxHead || DK == kMaxHead / 2) {  // fp32, 64- or 128-dim heads: every 16-byte load
                                                 // of the tile issued at once (DK / 4 per row)
      const int sh = DK == kMaxHead ? 5 : 4, msk = (1 << sh) - 1, nj = DK / 16;
      const float* kf = reinterpret_cast<const float*>(k);
      const float* qf = reinterpret_cast<const float*>(q);
      float4 kv[8], qv[8];
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i4 = tid + j * NT, t = i4 >> sh, d4 = (i4 & msk) * 4;
        const size_t off = ((size_t)(t0 + t) * p.h_k + hk) * DK + d4;
        const bool in = j < nj && t < n;
        kv[j] = in ? *reinterpret_cast<const float4*>(kf + off) : z4;
        qv[j] = (p.write_O && in) ? *reinterpret_cast<const float4*>(qf + off) : z4;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= nj) break;
        const int i4 = tid + j * NT, t = i4 >> sh, d4 = (i4 & msk) * 4;
        *reinterpret_cast<float4*>(sm.K + t * KST + d4) = kv[j];
        if (p.write_O) *reinterpret_cast<float4*>(sm.Q + t * KST + d4) = qv[j];
      }
      loaded = true;
    }
  }
  if (!loaded) {
#pragma unroll 8
    for (int i = tid; i < C * DK; i += NT) {
      const int t = i / DK, d = i % DK;
      const size_t off = ((size_t)(t0 + t) * p.h_k + hk) * DK + d;
      sm.K[t * KST + d] = t < n ? ld_in(k, off) : 0.f;
      if (p.write_O) sm.Q[t * KST + d] = t < n ? ld_in(q, off) : 0.f;
    }
  }
  if (tid < 2 * C) {  // gates of slot tid / 64
    const int sl = tid >> 6, t = tid & 63;
    const bool in = t < n && sl < nslots;
    sm.G[sl][t] = in ? p.g[(size_t)(t0 + t) * p.h_v + h0 + sl] : 0.f;
    sm.beta[sl][t] = in ? p.beta[(size_t)(t0 + t) * p.h_v + h0 + sl] : 0.f;
  }
  __syncthreads();
  // per-token L2 normalisation (q also takes the scale), gate prefix sums (warp 0: slot 0, warp 1: slot 1)
  for (int t = warp; t < C; t += NT / 32) {
    float sk = 0.f, sq = 0.f;
    for (int d = lane; d < DK; d += 32) {
      const float a = sm.K[t * KST + d];
      sk += a * a;
      if (p.write_O) { const float b = sm.Q[t * KST + d]; sq += b * b; }
    }
    for (int o = 16; o > 0; o >>= 1) {
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    const float fk = p.l2norm ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
    const float fq = (p.l2norm ? 1.f / sqrtf(sq + 1e-6f) : 1.f) * p.scale;
    for (int d = lane; d < DK; d += 32) {
      sm.K[t * KST + d] *= fk;
      if (p.write_O) sm.Q[t * KST + d] *= fq;
    }
    if (lane == 0) {
      sm.rk[t] = fk;
      sm.rq[t] = fq;
    }
  }
  if (warp < 2) {
    float a = sm.G[warp][lane], b = sm.G[warp][lane + 32];
    for (int o = 1; o < 32; o <<= 1) {
      const float xa = __shfl_up_sync(0xffffffffu, a, o);
      const float xb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) { a += xa; b += xb; }
    }
    b += __shfl_sync(0xffffffffu, a, 31);
    sm.G[warp][lane] = a;
    sm.G[warp][lane + 32] = b;
  }
  __syncthreads();
  {  // Gram matrices on warp-level tensor cores (split tf32), once for both slots; then per slot A
     // (strictly lower, gated, beta-weighted) into shared memory and P into the record (only when
     // outputs are wanted: the scan reads it for nothing else).
     // Warp w -> rows 16 (w % 4) + [0, 16), columns 32 (w / 4) + [0, 32).
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2), g = lane >> 2, q4 = lane & 3;
    float akk[4][4] = {}, aqk[4][4] = {};
    tcp::warp_mma_tf32x3<4>(akk, [&](int m, int kk) { return sm.K[m * KST + kk]; },
                            [&](int kk, int nn) { return sm.K[nn * KST + kk]; }, m0, n0, 0, DK, C);
    if (p.write_O)
      tcp::warp_mma_tf32x3<4>(aqk, [&](int m, int kk) { return sm.Q[m * KST + kk]; },
                              [&](int kk, int nn) { return sm.K[nn * KST + kk]; }, m0, n0, 0, DK, C);
    for (int sl = 0; sl < nslots; ++sl) {
      float* rec = rec_of(sl);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int t = m0 + g + 8 * hh, s0 = n0 + 8 * j + 2 * q4;
          float pv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int s = s0 + e;
            const float decay = s <= t ? expf(sm.G[sl][t] - sm.G[sl][s]) : 0.f;
            sm.A[sl][t * tcp::MST + s] =
                (s < t && !p.scalar_decay) ? sm.beta[sl][t] * decay * akk[j][2 * hh + e] : 0.f;
            pv[e] = s <= t ? decay * aqk[j][2 * hh + e] : 0.f;
          }
          if (p.write_O) *reinterpret_cast<float2*>(rec + REC_P + t * C + s0) = make_float2(pv[0], pv[1]);
        }
    }
  }
  __syncthreads();
  const int slot = warp >> 2, gt = tid & 127;  // warpgroup = v-head slot
  if (slot < nslots) tcp::invert_unit_lower(sm.A[slot], sm.M[slot], gt, 1 + slot);
  __syncthreads();
  for (int sl = 0; sl < nslots; ++sl) {
    float* rec = rec_of(sl);
    if (tid < C) {
      const int t = tid;
      const float Gl = sm.G[sl][C - 1];
      rec[REC_GAM + t] = expf(sm.G[sl][t]);
      rec[REC_WEND + t] = expf(Gl - sm.G[sl][t]);
      rec[REC_BETA + t] = sm.beta[sl][t];
      rec[REC_RK + t] = sm.rk[t];
      rec[REC_RQ + t] = sm.rq[t];
    }
    for (int i = tid; i < C * C / 4; i += NT) {
      const int t = i / (C / 4), s4 = (i % (C / 4)) * 4;
      *reinterpret_cast<float4*>(rec + REC_M + t * C + s4) = *reinterpret_cast<const float4*>(sm.M[sl] + t * tcp::MST + s4);
    }
  }
}

template <typename Tin>
__global__ void __launch_bounds__(NT) simt_chunk_scan_kernel(SimtParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const int slice = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int DK = p.d_k, DV = p.d_v;
  const int rows_total = DV + (p.augmented ? DK : 0);
  const int row0 = slice * RS;
  const int hk = h / (p.h_v / p.h_k);
  const Tin* __restrict__ q = static_cast<const Tin*>(p.q);
  const Tin* __restrict__ k = static_cast<const Tin*>(p.k);
  const Tin* __restrict__ v = static_cast<const Tin*>(p.v);

  // cu == nullptr: a single sequence covering every token
  // A malformed range (see chunk_info) is skipped and reported; in two-pass mode `first` is the
  // global index of this sequence's first chunk in the records.
  int first = 0;
  if (p.cu) {
    const tcp::ChunkInfo ci = tcp::chunk_info(p.cu, p.n_seqs, p.total_tokens, seq, -1, sm.scratch);
    if (!ci.valid) {
      if (tid == 0) atomicExch(p.status, GDN_ERR_SHAPE);
      return;
    }
    first = ci.first;
  }
  const int t_begin = p.cu ? p.cu[seq] : 0;
  const int t_end = p.cu ? p.cu[seq + 1] : p.total_tokens;

  // entering state of this slice
  for (int i = tid; i < RS * DK; i += NT) {
    const int r = i / DK, d = i % DK, rg = row0 + r;
    float s = 0.f;
    if (rg < DV) {
      if (p.S0) s = p.S0[(((size_t)seq * p.h_v + h) * DV + rg) * DK + d];
    } else if (rg < rows_total) {
      s = (d == rg - DV) ? 1.f : 0.f;
    }
    sm.S[r * KST + d] = s;
  }

  // fp32 inputs with 64- or 128-dim heads on the record path: each chunk's keys, M, value slice
  // and gate factors arrive by asynchronous copies issued one chunk (keys) or half a chunk (the
  // rest) ahead; the keys stay unscaled and their norm factors rk are applied to the products.
  // A row of keys (queries) is DK / 4 16-byte pieces: thread item i4 -> row i4 >> ksh.
  bool vec = false;
  if constexpr (sizeof(Tin) == 4) vec = p.rec && (DK == kMaxHead || DK == kMaxHead / 2) && (DV % RS == 0);
  const int ksh = DK == kMaxHead ? 5 : 4, kmask = (1 << ksh) - 1, nkj = DK / 16;
  const float* kf = reinterpret_cast<const float*>(k);
  const float* vf = reinterpret_cast<const float*>(v);
  auto rec_of = [&](int ck) {
    return reinterpret_cast<const float*>(p.rec) + ((size_t)(first + ck) * p.h_v + h) * REC_FLOATS;
  };
  auto pf_keys = [&](int t0c, int nc, float* kb) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= nkj) break;
      const int i4 = tid + j * NT, t = i4 >> ksh, d4 = (i4 & kmask) * 4;
      const bool ok = t < nc;
      cp_async16(kb + t * KST + d4, kf + ((size_t)(t0c + (ok ? t : 0)) * p.h_k + hk) * DK + d4, ok);
    }
  };
  auto pf_rest = [&](const float* Rc, int t0c, int nc) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = (tid + j * NT) * 4, t = i / C, s2 = i % C;
      cp_async16(sm.M + t * GST + s2, Rc + REC_M + i, true);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i4 = tid + j * NT, t = i4 >> 3, r4 = (i4 & 7) * 4;
      const bool ok = t < nc && row0 + r4 < DV;
      cp_async16(sm.V + t * VST + r4, ok ? vf + ((size_t)(t0c + t) * p.h_v + h) * DV + row0 + r4 : vf, ok);
    }
    if (tid < 64) cp_async16(sm.gam + tid * 4, Rc + REC_GAM + tid * 4, true);  // gam, wend, beta, rk
  };
  if (vec && t_begin < t_end) {
    pf_keys(t_begin, min(C, t_end - t_begin), sm.K);
    pf_rest(rec_of(0), t_begin, min(C, t_end - t_begin));
    cp_async_commit();
  }

  for (int t0 = t_begin, ck = 0; t0 < t_end; t0 += C, ++ck) {
    const int n = min(C, t_end - t0);
    const bool more = t0 + C < t_end;
    float* const Kc = (vec && (ck & 1)) ? sm.K2 : sm.K;  // this chunk's keys
    __syncthreads();
    if (p.rec) {
      // ---- chunk-shared quantities from the record; keys (and queries) scaled by their norms
      const float* R = rec_of(ck);
      if (vec) {
        cp_async_wait_all();
        if (p.write_O) {  // queries (scaled by rq) and P, read directly
          const float* qf = reinterpret_cast<const float*>(q);
          const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
          float4 qv[8], pv[4];
          float rqv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i4 = tid + j * NT, t = i4 >> ksh, d4 = (i4 & kmask) * 4;
            const bool in = j < nkj && t < n;
            qv[j] = in ? *reinterpret_cast<const float4*>(qf + ((size_t)(t0 + t) * p.h_k + hk) * DK + d4) : z4;
            rqv[j] = j < nkj ? R[REC_RQ + t] : 0.f;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) pv[j] = *reinterpret_cast<const float4*>(R + REC_P + (tid + j * NT) * 4);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j >= nkj) break;
            const int i4 = tid + j * NT, t = i4 >> ksh, d4 = (i4 & kmask) * 4;
            float* qd = sm.Q + t * KST + d4;
            qd[0] = rqv[j] * qv[j].x; qd[1] = rqv[j] * qv[j].y; qd[2] = rqv[j] * qv[j].z; qd[3] = rqv[j] * qv[j].w;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = (tid + j * NT) * 4, t = i / C, s2 = i % C;
            float* pd = sm.P + t * GST + s2;
            pd[0] = pv[j].x; pd[1] = pv[j].y; pd[2] = pv[j].z; pd[3] = pv[j].w;
          }
        }
        __syncthreads();  // this chunk's copies (issued by every thread) have all landed
        if (more) {
          pf_keys(t0 + C, min(C, t_end - t0 - C), (ck & 1) ? sm.K : sm.K2);
          cp_async_commit();
        }
      } else {
#pragma unroll 8
      for (int i = tid; i < C * DK; i += NT) {
        const int t = i / DK, d = i % DK;
        const size_t off = ((size_t)(t0 + t) * p.h_k + hk) * DK + d;
        sm.K[t * KST + d] = t < n ? R[REC_RK + t] * ld_in(k, off) : 0.f;
        if (p.write_O) sm.Q[t * KST + d] = t < n ? R[REC_RQ + t] * ld_in(q, off) : 0.f;
      }
      for (int i = tid; i < C * RS; i += NT) {
        const int t = i / RS, r = i % RS, rg = row0 + r;
        float x = 0.f;
        if (t < n && rg < DV) x = ld_in(v, ((size_t)(t0 + t) * p.h_v + h) * DV + rg);
        sm.V[t * VST + r] = x;
      }
#pragma unroll 8
      for (int i = tid; i < C * C; i += NT) {
        const int t = i / C, s2 = i % C;
        sm.M[t * GST + s2] = R[REC_M + i];
        if (p.write_O) sm.P[t * GST + s2] = R[REC_P + i];
      }
      if (tid < C) {  // keys stored scaled: rk = 1
        sm.gam[tid] = R[REC_GAM + tid];
        sm.wend[tid] = R[REC_WEND + tid];
        sm.beta[tid] = R[REC_BETA + tid];
        sm.rk[tid] = 1.f;
      }
      __syncthreads();
      }
      {  // X = diag(rk) K S0^T (64 x 32, K = d_k): warp w -> rows 16 (w / 2), columns 16 (w % 2) + [0, 16)
        const int w = tid >> 5, lane = tid & 31, m0 = 16 * (w >> 1), n0 = 16 * (w & 1);
        float acc[2][4] = {};
        tcp::warp_mma_tf32x3<2>(acc, [&](int m, int kk) { return Kc[m * KST + kk]; },
                                [&](int kk, int nn) { return sm.S[nn * KST + kk]; }, m0, n0, 0, DK, RS);
        const float ra = sm.rk[m0 + (lane >> 2)], rb = sm.rk[m0 + (lane >> 2) + 8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc[j][0] *= ra; acc[j][1] *= ra; acc[j][2] *= rb; acc[j][3] *= rb;
        }
        store_tile(sm.X, VST, acc, m0, n0, lane);
      }
      __syncthreads();
    } else {
    // ---- load the chunk
    for (int i = tid; i < C * DK; i += NT) {
      const int t = i / DK, d = i % DK;
      const size_t off = ((size_t)(t0 + t) * p.h_k + hk) * DK + d;
      sm.K[t * KST + d] = t < n ? ld_in(k, off) : 0.f;
      if (p.write_O) sm.Q[t * KST + d] = t < n ? ld_in(q, off) : 0.f;
    }
    for (int i = tid; i < C * RS; i += NT) {
      const int t = i / RS, r = i % RS, rg = row0 + r;
      float x = 0.f;
      if (t < n && rg < DV) x = ld_in(v, ((size_t)(t0 + t) * p.h_v + h) * DV + rg);
      sm.V[t * VST + r] = x;
    }
    if (tid < C) {
      const bool in = tid < n;
      sm.G[tid] = in ? p.g[(size_t)(t0 + tid) * p.h_v + h] : 0.f;
      sm.beta[tid] = in ? p.beta[(size_t)(t0 + tid) * p.h_v + h] : 0.f;
      sm.rk[tid] = 1.f;  // keys are normalised in place below
    }
    __syncthreads();

    // ---- per-token L2 normalisation (and q scale), gate prefix sums
    {
      const int warp = tid / 32, lane = tid % 32;
      for (int t = warp; t < C; t += NT / 32) {
        float sk = 0.f, sq = 0.f;
        for (int d = lane; d < DK; d += 32) {
          const float a = sm.K[t * KST + d];
          sk += a * a;
          if (p.write_O) { const float b = sm.Q[t * KST + d]; sq += b * b; }
        }
        for (int o = 16; o > 0; o >>= 1) {
          sk += __shfl_xor_sync(0xffffffffu, sk, o);
          sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        const float fk = p.l2norm ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
        const float fq = (p.l2norm ? 1.f / sqrtf(sq + 1e-6f) : 1.f) * p.scale;
        for (int d = lane; d < DK; d += 32) {
          sm.K[t * KST + d] *= fk;
          if (p.write_O) sm.Q[t * KST + d] *= fq;
        }
      }
      if (warp == 0) {
        float a = sm.G[lane], b = sm.G[lane + 32];
        for (int o = 1; o < 32; o <<= 1) {
          const float xa = __shfl_up_sync(0xffffffffu, a, o);
          const float xb = __shfl_up_sync(0xffffffffu, b, o);
          if (lane >= o) { a += xa; b += xb; }
        }
        b += __shfl_sync(0xffffffffu, a, 31);
        sm.G[lane] = a;
        sm.G[lane + 32] = b;
        sm.gam[lane] = expf(a);
        sm.gam[lane + 32] = expf(b);
        const float Gl = __shfl_sync(0xffffffffu, b, 31);
        sm.wend[lane] = expf(Gl - a);
        sm.wend[lane + 32] = expf(Gl - b);
      }
    }
    __syncthreads();

    // ---- Gram matrices: A (strictly lower, gated, beta-weighted) and P (inclusive lower, gated)
    {
      const int ti = (tid / 16) * 4, si = (tid % 16) * 4;
      float akk[4][4] = {}, aqk[4][4] = {};
      for (int d = 0; d < DK; ++d) {
        float a[4], b[4], c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[i] = sm.K[(ti + i) * KST + d];
          b[i] = sm.K[(si + i) * KST + d];
          c[i] = p.write_O ? sm.Q[(ti + i) * KST + d] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            akk[i][j] = fmaf(a[i], b[j], akk[i][j]);
            aqk[i][j] = fmaf(c[i], b[j], aqk[i][j]);
          }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = ti + i, s = si + j;
          const float decay = s <= t ? expf(sm.G[t] - sm.G[s]) : 0.f;
          sm.A[t * GST + s] = (s < t && !p.scalar_decay) ? sm.beta[t] * decay * akk[i][j] : 0.f;
          sm.P[t * GST + s] = s <= t ? decay * aqk[i][j] : 0.f;
        }
    }
    __syncthreads();

    // ---- M = (I + A)^{-1} by forward substitution, one column per thread (warps 0-1);
    //      meanwhile X = K S0^T (warps 2-7)
    if (tid < C) {
      const int j = tid;
      for (int t = 0; t < C; ++t) {
        float m;
        if (t < j) m = 0.f;
        else if (t == j) m = 1.f;
        else {
          float acc0 = 0.f, acc1 = 0.f;
          int s = j;
          for (; s + 1 < t; s += 2) {
            acc0 = fmaf(sm.A[t * GST + s], sm.M[s * GST + j], acc0);
            acc1 = fmaf(sm.A[t * GST + s + 1], sm.M[(s + 1) * GST + j], acc1);
          }
          if (s < t) acc0 = fmaf(sm.A[t * GST + s], sm.M[s * GST + j], acc0);
          m = -(acc0 + acc1);
        }
        sm.M[t * GST + j] = m;
      }
    } else {
      for (int i = tid - C; i < C * RS; i += NT - C) {
        const int t = i / RS, r = i % RS;
        float acc = 0.f;
        for (int d = 0; d < DK; ++d) acc = fmaf(sm.K[t * KST + d], sm.S[r * KST + d], acc);
        sm.X[t * VST + r] = acc;
      }
    }
    __syncthreads();
    }

    // ---- R = diag(beta) (V - diag(gamma) X)   (in place in V)
    for (int i = tid; i < C * RS; i += NT) {
      const int t = i / RS, r = i % RS;
      // (scalar-decay family: no rank-1 projection, so no correction by the entering state)
      sm.V[t * VST + r] = sm.beta[t] * (p.scalar_decay ? sm.V[t * VST + r] : sm.V[t * VST + r] - sm.gam[t] * sm.X[t * VST + r]);
    }
    __syncthreads();

    // ---- U = M R into X (M lower triangular), and diag(wend rk) U into the A area (free once M
    //      is known) for the state update
    {
      const int w = tid >> 5, lane = tid & 31, m0 = 16 * (w >> 1), n0 = 16 * (w & 1);
      float acc[2][4] = {};
      tcp::warp_mma_tf32x3<2>(acc, [&](int m, int kk) { return sm.M[m * GST + kk]; },
                              [&](int kk, int nn) { return sm.V[kk * VST + nn]; }, m0, n0, 0, m0 + 16, RS);
      store_tile(sm.X, VST, acc, m0, n0, lane);
      const float wa = sm.wend[m0 + (lane >> 2)] * sm.rk[m0 + (lane >> 2)];
      const float wb = sm.wend[m0 + (lane >> 2) + 8] * sm.rk[m0 + (lane >> 2) + 8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[j][0] *= wa; acc[j][1] *= wa; acc[j][2] *= wb; acc[j][3] *= wb;
      }
      store_tile(sm.A, VST, acc, m0, n0, lane);
    }
    __syncthreads();

    // ---- outputs O = diag(gamma) Q S0^T + P U (P lower triangular)
    if (p.write_O) {
      Tin* O = static_cast<Tin*>(p.O);
      const int w = tid >> 5, lane = tid & 31, m0 = 16 * (w >> 1), n0 = 16 * (w & 1);
      const int g = lane >> 2, q4 = lane & 3;
      float acc[2][4] = {};
      tcp::warp_mma_tf32x3<2>(acc, [&](int m, int kk) { return sm.Q[m * KST + kk]; },
                              [&](int kk, int nn) { return sm.S[nn * KST + kk]; }, m0, n0, 0, DK, RS);
      const float ga = sm.gam[m0 + g], gb = sm.gam[m0 + g + 8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[j][0] *= ga; acc[j][1] *= ga; acc[j][2] *= gb; acc[j][3] *= gb;
      }
      tcp::warp_mma_tf32x3<2>(acc, [&](int m, int kk) { return sm.P[m * GST + kk]; },
                              [&](int kk, int nn) { return sm.X[kk * VST + nn]; }, m0, n0, 0, m0 + 16, RS);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = m0 + g + 8 * (e >> 1), rg = row0 + n0 + 8 * j + 2 * q4 + (e & 1);
          if (t < n && rg < DV) st_out(O, ((size_t)(t0 + t) * p.h_v + h) * DV + rg, acc[j][e]);
        }
    }
    const float gC = sm.gam[C - 1];
    if (vec && more) {  // the next chunk's M, value slice and factors: their current readers are done
      __syncthreads();
      pf_rest(rec_of(ck + 1), t0 + C, min(C, t_end - t0 - C));
      cp_async_commit();
    }
    // ---- new state: S <- gamma_C S + (diag(wend rk) U)^T K (32 x d_k, K = 64 tokens):
    //      warp w -> rows 16 (w / 4), columns 32 (w % 4) + [0, 32)
    {
      const int w = tid >> 5, lane = tid & 31, m0 = 16 * (w >> 2), n0 = 32 * (w & 3);
      const int g = lane >> 2, q4 = lane & 3;
      float acc[4][4] = {};
      tcp::warp_mma_tf32x3<4>(acc, [&](int m, int kk) { return sm.A[kk * VST + m]; },
                              [&](int kk, int nn) { return Kc[kk * KST + nn]; }, m0, n0, 0, C, DK);
      __syncthreads();  // every read of the entering state (X, outputs) is done
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int d = n0 + 8 * j + 2 * q4;
        if (d >= DK) continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float* sp = &sm.S[(m0 + g + 8 * (e >> 1)) * KST + d + (e & 1)];
          *sp = fmaf(gC, *sp, acc[j][e]);
        }
      }
    }
  }
  __syncthreads();

  // ---- final state: value rows to S_out, transition rows (P = T_C^T) to T_out transposed
  for (int i = tid; i < RS * DK; i += NT) {
    const int r = i / DK, d = i % DK, rg = row0 + r;
    const float s = sm.S[r * KST + d];
    if (rg < DV) {
      p.S_out[(((size_t)seq * p.h_v + h) * DV + rg) * DK + d] = s;
    } else if (rg < rows_total) {
      const int pr = rg - DV;  // P[pr][d] = T_C[d][pr]
      p.T_out[(((size_t)seq * p.h_v + h) * DK + d) * DK + pr] = s;
    }
  }
}

}  // namespace

cudaError_t launch_replay_simt(const SimtParams& p, int bf16, cudaStream_t stream) {
  if (p.n_seqs == 0) return cudaSuccess;
  const int rows = p.d_v + (p.augmented ? p.d_k : 0);
  dim3 grid((rows + RS - 1) / RS, p.h_v, p.n_seqs);
  const size_t smem = sizeof(Smem);
  cudaError_t e;
  if (bf16) {
    e = cudaFuncSetAttribute(simt_chunk_scan_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    simt_chunk_scan_kernel<__nv_bfloat16><<<grid, NT, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(simt_chunk_scan_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    simt_chunk_scan_kernel<float><<<grid, NT, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

size_t simt_records_bytes(int n_seqs, int total_tokens, int h_v) {
  const size_t chunks = (size_t)tcp::chunks_of(total_tokens) + (size_t)n_seqs;  // >= sum of ceil(len / 64)
  return chunks * (size_t)h_v * REC_FLOATS * sizeof(float);
}

cudaError_t launch_replay_simt_two_pass(SimtParams p, int bf16, void* workspace, size_t bytes, cudaStream_t stream) {
  if (p.n_seqs == 0) return cudaSuccess;
  if (!workspace || bytes < simt_records_bytes(p.n_seqs, p.total_tokens, p.h_v)) return cudaErrorInvalidValue;
  p.rec = static_cast<unsigned char*>(workspace);
  const int chunks_ub = tcp::chunks_of(p.total_tokens) + (p.cu ? p.n_seqs : 0);
  if (p.total_tokens > 0) {
    const int G = p.h_v / p.h_k;
    const dim3 grid(chunks_ub, p.h_k * ((G + 1) / 2));  // (chunk, key head, pair of its v-heads)
    const size_t smem = p.write_O ? sizeof(PrepSmem) : kPrepSmemNoQ;
    cudaError_t e;
    if (bf16) {
      e = cudaFuncSetAttribute(simt_chunk_prep_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
      simt_chunk_prep_kernel<__nv_bfloat16><<<grid, NT, smem, stream>>>(p);
    } else {
      e = cudaFuncSetAttribute(simt_chunk_prep_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      simt_chunk_prep_kernel<float><<<grid, NT, smem, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // state only, 128-dim heads: the tensor-core scan over the same records (fp32 accuracy)
  if (chunkop_tc_supported(p, bf16)) return launch_chunkop_tc(p, bf16, stream);
  return launch_replay_simt(p, bf16, stream);
}

}  // namespace gdn
