/*
 * gdn.h -- C ABI of libgdn.so: the Gated DeltaNet tail-replay state rebuild
 * on one GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 * State layout.  A recurrent state S is fp32, d_v x d_k, row-major, and one
 * token updates it as
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   alpha_t = exp(g_t),
 * which is Eq. (1) of "Tail-Replay: Escaping the Curse of Linear Attention in
 * Prefix Caching for Hybrid LLMs" (section 2) written on the transposed state
 * (T_t = alpha_t (I - beta_t k_t k_t^T) is symmetric, so T_t S^T = (S T_t)^T).
 * The readout is o_t = S_t (scale * q_t) with the updated state.
 *
 * Token-major inputs.  q, k: [total_tokens][h_k][d_k]; v and O: [total_tokens]
 * [h_v][d_v]; g and beta: fp32 [total_tokens][h_v].  Sequences (replay tails)
 * are packed back to back; cu_seqlens (int32, DEVICE memory, n_seqs + 1
 * entries, non-decreasing, cu_seqlens[n_seqs] <= total_tokens) gives each
 * one's token range.  A range that breaks this (negative, past total_tokens,
 * or starting before an earlier offset) is skipped, its state left untouched,
 * and reported as GDN_ERR_SHAPE through gdn_get_status.  v-head h reads q/k
 * head h / (h_v / h_k) (consecutive v-heads share a key head).  States: fp32 [n_seqs][h_v][d_v][d_k].
 *
 * Ownership and memory.  Every pointer except the host arrays of gdn_compose
 * is a DEVICE pointer owned by the caller; the library never frees or keeps
 * them.  Calls that need scratch memory take it from a per-device pool that
 * the library grows on first need with cudaMallocAsync on the caller's
 * stream (stream-ordered) and keeps until process exit.
 *
 * Asynchrony and errors.  Every call only enqueues work on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and returns 0 (GDN_OK) or a
 * negative GDN_ERR_* code without launching anything.  No exception crosses
 * the ABI.  gdn_last_error() gives a thread-local message for the last
 * failure.  Errors found on the device (malformed cu_seqlens) are recorded in
 * a sticky per-device status word that gdn_get_status() returns and clears.
 *
 * Alignment.  q, k, v, O, S0, S_out, T and S_local base pointers must be
 * 16-byte aligned; g, beta and cu_seqlens 4-byte aligned (else GDN_ERR_ALIGN).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

/* return codes */
#define GDN_OK 0
#define GDN_ERR_ARG (-1)         /* null pointer, negative size, bad flag */
#define GDN_ERR_SHAPE (-2)       /* inconsistent sizes (h_v % h_k, token ranges) */
#define GDN_ERR_ALIGN (-3)       /* a base pointer breaks the alignment rule */
#define GDN_ERR_UNSUPPORTED (-4) /* a head size or dtype the library has no kernel for */
#define GDN_ERR_CUDA (-5)        /* a CUDA runtime call failed (message in gdn_last_error) */
#define GDN_ERR_TIMEOUT (-6)     /* a bounded device-side wait gave up */
#define GDN_ERR_NOMEM (-7)       /* the scratch pool could not grow */

/* storage type of q, k, v and O (g, beta and every state are always fp32) */
#define GDN_F32 0
#define GDN_BF16 1

/* flags */
#define GDN_QK_L2NORM 1u   /* normalise q and k per (token, head): x / sqrt(sum x^2 + 1e-6) */
#define GDN_STATE_ONLY 2u  /* rebuild the state only; O_out may be NULL and is not written */
#define GDN_PRECISE 4u     /* bf16 inputs: take the fp32-accurate path (as fp32 inputs do) */
/* Scalar-decay recurrence family (Mamba-2), which "LinearKV: One Cached State
 * Suffices for Position-Independent Caching in Hybrid LLMs" (composition passage)
 * sets beside GDN: the per-token transition is the scalar alpha_t instead of
 * alpha_t (I - beta_t k_t k_t^T), i.e. S_t = alpha_t S_{t-1} + beta_t v_t k_t^T
 * (beta_t scales the input; same readout), so a chunk's transition is
 * (prod alpha_t) I.  Accepted by gdn_replay, gdn_replay_noalloc and
 * gdn_chunk_operator (whose T_out is then that scaled identity). */
#define GDN_SCALAR_DECAY 8u

typedef struct {
  int32_t n_seqs;       /* packed sequences (replay tails, or chunks for gdn_chunk_operator) */
  int32_t total_tokens; /* rows of q, k, v, g, beta, O */
  int32_t h_k;          /* q/k heads */
  int32_t h_v;          /* v heads, a multiple of h_k */
  int32_t d_k;          /* key/query head dim: a multiple of 8, at most 128 */
  int32_t d_v;          /* value head dim: a multiple of 8, at most 128 */
  int32_t dtype;        /* GDN_F32 or GDN_BF16 */
  uint32_t flags;       /* GDN_QK_L2NORM | GDN_STATE_ONLY | GDN_PRECISE | GDN_SCALAR_DECAY */
  float scale;          /* multiplies q in the readout (1.0 when unsure) */
} gdn_dims;

/*
 * gdn_replay -- rebuild each sequence's recurrent state by replaying its tail.
 * Source: "Tail-Replay: ..." section 3, Eq. (2): the state at the start of
 * the tail is S0 (zero when S0 == NULL, the method's zero-initialised
 * replay), Eq. (1) is applied to every tail token, the final state is
 * written to S_out and, unless GDN_STATE_ONLY, every token's readout to O_out.
 *   q, k, v      inputs in `dims->dtype`, layouts above
 *   g, beta      fp32 [total_tokens][h_v]; g = log(alpha) <= 0
 *   cu_seqlens   int32 device [n_seqs + 1]
 *   S0           fp32 [n_seqs][h_v][d_v][d_k] or NULL
 *   O_out        [total_tokens][h_v][d_v] in `dims->dtype`; NULL iff GDN_STATE_ONLY.
 *                Rows outside every sequence's range are not written.
 *   S_out        fp32 [n_seqs][h_v][d_v][d_k]; may alias S0 (in-place update)
 * Computation: chunks of 64 tokens, fp32 state carried between chunks.  bf16
 * inputs with 128-dim heads run on the tcgen05 tensor cores; with several tails
 * their sequential scans start longest first (a small kernel ranks the tails by
 * length on the stream before the chunk kernels).  GDN_STATE_ONLY calls of that
 * kind with few enough (tail, head) pairs to give every 32-row slice of every
 * state its own SM carry the state through each chunk's d_k x d_k operator,
 * built ahead of the carry, so that the chunk-to-chunk chain is one product per
 * chunk; the result is the same state to rounding.  fp32 inputs,
 * other head sizes and GDN_PRECISE take the fp32-accurate path: fp32 data,
 * every contraction as three tf32 products (about 21 significant bits), in two
 * passes with pool scratch of (ceil(total_tokens / 64) + n_seqs) * h_v * 34048
 * bytes (gdn_workspace_bytes gives the amount); its second pass runs on the
 * tcgen05 tensor cores for state-only calls with 128-dim heads, on warp-level
 * tensor cores otherwise.
 */
int gdn_replay(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
               const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out, float* S_out,
               void* stream);

/*
 * gdn_replay_noalloc -- gdn_replay without any device allocation.
 * The pages have no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory when they call it, for example a
 * serving process that reserves almost all of the GPU's memory at start-up
 * (for its cache) and forbids allocations afterwards, or a caller whose
 * process-wide policy routes every device allocation through its own
 * allocator.  gdn_replay takes its scratch from a pool that can grow; this
 * variant instead uses one static device array of 96 MiB that every GPU that
 * loads the library holds until the process exits.
 *   Arguments, layouts, results and error codes are those of gdn_replay.
 *   Limit: the tensor-core path needs (ceil(total_tokens / 64) + n_seqs) * h_v
 *   * 41984 bytes of scratch, plus 4 * n_seqs bytes when n_seqs > 1
 *   (gdn_workspace_bytes gives the exact figure; a 3277-token tail at 32
 *   v-heads needs 67.9 MiB); a larger problem is rejected with GDN_ERR_NOMEM
 *   before anything is launched.  fp32 inputs and GDN_PRECISE need no scratch.
 *   Every call looks up the static array's device address (cudaGetSymbolAddress,
 *   with the caller's current device); the first lookup on a device can load
 *   the library's device code, so make the first call before any stream
 *   capture.
 *   All calls share the one array: calls that overlap on the GPU (on two
 *   streams, or from two threads) race with each other and must be serialised
 *   by the caller.  Every byte a call reads from the array is written by the
 *   same call first, so nothing needs clearing between calls.
 */
int gdn_replay_noalloc(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out, float* S_out,
                       void* stream);

/*
 * gdn_chunk_operator -- the affine operator of isolated chunks.
 * Source: "LinearKV: One Cached State Suffices for Position-Independent
 * Caching in Hybrid LLMs", composition passage: a chunk maps an entering
 * state to T_C S_in + S_local (transposed-state form), T_C the product of its
 * per-token transitions T_t = alpha_t (I - beta_t k_t k_t^T), latest on the
 * left, and S_local the state it reaches from an empty start.
 *   Each of the n_seqs ranges of cu_seqlens is one chunk (any length).  When
 *   cu_seqlens == NULL, n_seqs must be 1 and the chunk is all total_tokens.
 *   T_out       fp32 [n_seqs][h_v][d_k][d_k], T_C row-major, so that
 *               S_out = S_in T_C^T + S_local in this ABI's state layout
 *   Slocal_out  fp32 [n_seqs][h_v][d_v][d_k]
 * q is not needed; dims->scale and GDN_STATE_ONLY are ignored.  Computed at
 * fp32 accuracy whatever the input dtype, in two passes: the chunk-shared
 * quantities ((I + A)^{-1}, gates, norms) once per (64-token piece, v-head)
 * into pool scratch of (ceil(total_tokens / 64) + n_seqs) * h_v * 34048 bytes,
 * then the 128-row slices of the augmented state [S; P] (P seeded with the
 * identity, fed zero values; P = T_C^T after the chunk).  With d_k = d_v = 128
 * the second pass runs on the tensor cores (every contraction as three tf32
 * products); other head sizes take the fp32 CUDA-core path.
 */
int gdn_chunk_operator(const gdn_dims* dims, const void* k, const float* g, const float* beta, const void* v,
                       const int32_t* cu_seqlens, float* T_out, float* Slocal_out, void* stream);

/*
 * gdn_compose -- apply K chunk operators back to back.
 * Source: "LinearKV: ..." composition passage: the closed form
 * S_K = T_{C_K}...T_{C_2} S_local_1 + ... + T_{C_K} S_local_{K-1} + S_local_K
 * (transposed-state form), extended by T_{C_K}...T_{C_1} S_in when an
 * entering state is given.  Evaluated as S <- S T_j^T + S_local_j, j = 1..K.
 *   dims        uses h_v, d_k, d_v only (one state per v-head)
 *   K           number of chunks, 0 <= K <= 256
 *   T, Slocal   HOST arrays of K device pointers; T[j] fp32 [h_v][d_k][d_k],
 *               Slocal[j] fp32 [h_v][d_v][d_k]
 *   S_in        fp32 [h_v][d_v][d_k] or NULL (empty entering state)
 *   S_out       fp32 [h_v][d_v][d_k]; must not alias any input
 * With d_k = d_v = 128 the tensor cores do the products (T and S each split
 * into a tf32 part and an exact fp32 remainder; three products per step,
 * fp32 accuracy).  When the T[j] sit at one non-negative stride that is a
 * multiple of 512 bytes (e.g. the K slices of one [K][h_v][d_k][d_k] array)
 * each step's T arrives by tensor copies shared across the four CTAs of a
 * head; other pointer arrays take a slower path that copies T row by row.
 * Both give the same results up to fp32 rounding order.
 */
int gdn_compose(const gdn_dims* dims, int32_t K, const float* const* T, const float* const* Slocal,
                const float* S_in, float* S_out, void* stream);

/*
 * gdn_get_status -- synchronise `stream`, then return and clear the sticky
 * device status of the current device: GDN_OK, GDN_ERR_SHAPE (a malformed
 * cu_seqlens was skipped), GDN_ERR_TIMEOUT, or GDN_ERR_CUDA when the stream
 * itself reports an error.
 */
int gdn_get_status(void* stream);

/* Thread-local message of the last failed call ("" if none). */
const char* gdn_last_error(void);

/* Bytes of scratch the library's pool needs for this problem (0 if none). */
size_t gdn_workspace_bytes(const gdn_dims* dims);

/*
 * gdn_set_stage_event -- measurement hook (no counterpart on the pages).
 * `event` is a cudaEvent_t created by the caller.  The next gdn_replay or
 * gdn_replay_noalloc call made by this thread on the tensor-core path records
 * it on its stream between its two kernels (chunk prep, then scan), so that
 * the caller can time each kernel with its own events before and after the
 * call; the hook is then cleared.  Other calls ignore it.
 */
void gdn_set_stage_event(void* event);

/*
 * gdn_set_wait_limit_ns -- test hook for the device-side timeout path (no
 * counterpart on the pages).  Every wait inside the tensor-core kernels is
 * bounded (2 s by default): a wait that runs out makes the kernel stop issuing
 * work, let what it has already issued finish, and report GDN_ERR_TIMEOUT
 * through gdn_get_status, leaving the context usable.  The next gdn_compose
 * call made by this thread uses `ns` as that bound (0: a wait gives up unless
 * its event has already happened, so the call reports a timeout); the hook is
 * then cleared.  Results of a call that timed out are unspecified.
 */
void gdn_set_wait_limit_ns(uint64_t ns);

/* GDN_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
