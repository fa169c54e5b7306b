// C ABI of libgdn.so: argument checks, dispatch to the kernels, status word.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <cstdarg>
#include <mutex>
#include <string>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

thread_local std::string g_last_error;
thread_local void* g_stage_event = nullptr;  // cudaEvent_t to record between prep and scan, once
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
thread_local unsigned long long g_wait_ns = kDefaultWaitNs;  // next compose call's wait limit, once

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

__device__ int g_status;  // sticky per-device status (one copy per device that loads the library)

int check_head_dims(const gdn_dims* d) {
  if (d->h_k <= 0 || d->h_v <= 0) return fail(GDN_ERR_ARG, "h_k and h_v must be positive");
  if (d->h_v % d->h_k != 0) return fail(GDN_ERR_SHAPE, "h_v (%d) must be a multiple of h_k (%d)", d->h_v, d->h_k);
  if (d->d_k <= 0 || d->d_v <= 0 || d->d_k > kMaxHead || d->d_v > kMaxHead || d->d_k % 8 || d->d_v % 8)
    return fail(GDN_ERR_UNSUPPORTED, "d_k=%d, d_v=%d: need multiples of 8 in [8, %d]", d->d_k, d->d_v, kMaxHead);
  return GDN_OK;
}

int check_token_dims(const gdn_dims* d) {
  if (d->n_seqs < 0 || d->total_tokens < 0) return fail(GDN_ERR_ARG, "negative n_seqs or total_tokens");
  if (d->dtype != GDN_F32 && d->dtype != GDN_BF16) return fail(GDN_ERR_UNSUPPORTED, "dtype %d", d->dtype);
  if (d->flags & ~(GDN_QK_L2NORM | GDN_STATE_ONLY | GDN_PRECISE | GDN_SCALAR_DECAY))
    return fail(GDN_ERR_ARG, "unknown flag bits 0x%x", d->flags);
  return check_head_dims(d);
}

// Stream-ordered scratch: one private memory pool per device that keeps its memory
// (release threshold = max), so after the first call allocations are pool hits.
int scratch_pool(cudaMemPool_t* out) {
  static std::mutex mu;
  static cudaMemPool_t pools[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(GDN_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&pools[dev], &props);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = UINT64_MAX;
    e = cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolSetAttribute");
  }
  *out = pools[dev];
  return GDN_OK;
}

}  // namespace

// Argument checks of gdn_replay and gdn_replay_noalloc (one set of rules for both): fills *p,
// sets *nothing_to_do for an empty batch.
int check_replay_args(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out, float* S_out,
                      SimtParams* p, bool* nothing_to_do) {
  g_last_error.clear();
  *nothing_to_do = false;
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  int rc = check_token_dims(dims);
  if (rc) return rc;
  const bool state_only = dims->flags & GDN_STATE_ONLY;
  if (dims->n_seqs == 0) {
    *nothing_to_do = true;
    return GDN_OK;
  }
  if (!cu_seqlens || !S_out) return fail(GDN_ERR_ARG, "cu_seqlens and S_out are required");
  if (!state_only && !O_out) return fail(GDN_ERR_ARG, "O_out is NULL without GDN_STATE_ONLY");
  if (dims->total_tokens > 0 && (!q || !k || !v || !g || !beta))
    return fail(GDN_ERR_ARG, "q, k, v, g and beta are required when total_tokens > 0");
  const void* p16[] = {q, k, v, O_out, S0, S_out};
  for (const void* ptr : p16)
    if (ptr && !aligned(ptr, 16)) return fail(GDN_ERR_ALIGN, "q, k, v, O, S0 and S_out must be 16-byte aligned");
  if (!aligned(g, 4) || !aligned(beta, 4) || !aligned(cu_seqlens, 4))
    return fail(GDN_ERR_ALIGN, "g, beta and cu_seqlens must be 4-byte aligned");
  int* status = device_status_word();
  if (!status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  *p = SimtParams{};
  p->q = q; p->k = k; p->v = v; p->g = g; p->beta = beta; p->cu = cu_seqlens; p->S0 = S0;
  p->O = state_only ? nullptr : O_out;
  p->S_out = S_out; p->T_out = nullptr;
  p->n_seqs = dims->n_seqs; p->total_tokens = dims->total_tokens;
  p->h_k = dims->h_k; p->h_v = dims->h_v; p->d_k = dims->d_k; p->d_v = dims->d_v;
  p->augmented = 0; p->l2norm = (dims->flags & GDN_QK_L2NORM) ? 1 : 0;
  p->write_O = state_only ? 0 : 1; p->scale = dims->scale; p->status = status;
  p->scalar_decay = (dims->flags & GDN_SCALAR_DECAY) ? 1 : 0;
  return GDN_OK;
}

int report_error(int code, const char* message) { return fail(code, "%s", message); }

void* take_stage_event() {
  void* e = g_stage_event;
  g_stage_event = nullptr;
  return e;
}

unsigned long long take_wait_limit_ns() {
  const unsigned long long ns = g_wait_ns;
  g_wait_ns = kDefaultWaitNs;
  return ns;
}

int* device_status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

void gdn_set_stage_event(void* event) { g_stage_event = event; }

void gdn_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns; }

const char* gdn_last_error(void) { return g_last_error.c_str(); }

size_t gdn_workspace_bytes(const gdn_dims* dims) {
  if (!dims || dims->total_tokens <= 0 || dims->n_seqs <= 0 || dims->h_v <= 0) return 0;
  if (dims->dtype == GDN_BF16 && !(dims->flags & GDN_PRECISE) && dims->d_k == kMaxHead && dims->d_v == kMaxHead)
    return replay_tc_workspace_bytes(dims->n_seqs, dims->total_tokens, dims->h_v);
  return simt_records_bytes(dims->n_seqs, dims->total_tokens, dims->h_v);  // fp32 path: its records
}

int gdn_replay(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
               const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out, float* S_out,
               void* stream) {
  SimtParams p;
  bool nothing = false;
  const int rc = check_replay_args(dims, q, k, v, g, beta, cu_seqlens, S0, O_out, S_out, &p, &nothing);
  if (rc || nothing) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dims->dtype == GDN_BF16 && !(dims->flags & GDN_PRECISE) && replay_tc_supported(p)) {
    const size_t bytes = replay_tc_workspace_bytes(p.n_seqs, p.total_tokens, p.h_v);
    cudaMemPool_t pool = nullptr;
    int prc = scratch_pool(&pool);
    if (prc) return prc;
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, st);
    if (e != cudaSuccess) return fail(GDN_ERR_NOMEM, "scratch of %zu bytes: %s", bytes, cudaGetErrorString(e));
    e = launch_replay_tc(p, ws, bytes, st);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_replay tensor-core launch");
    if (ef != cudaSuccess) return cuda_fail(ef, "scratch release");
    return GDN_OK;
  }
  // fp32 path in two passes: the chunk-shared quantities (norms, gates, (I + A)^{-1}, P) once per
  // (chunk, v-head) into pool scratch, then the row slices of each state read them.
  const size_t bytes = simt_records_bytes(p.n_seqs, p.total_tokens, p.h_v);
  cudaMemPool_t pool = nullptr;
  int prc = scratch_pool(&pool);
  if (prc) return prc;
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, st);
  if (e != cudaSuccess) return fail(GDN_ERR_NOMEM, "scratch of %zu bytes: %s", bytes, cudaGetErrorString(e));
  e = launch_replay_simt_two_pass(p, dims->dtype == GDN_BF16, ws, bytes, st);
  const cudaError_t ef = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, "gdn_replay launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch release");
  return GDN_OK;
}

int gdn_chunk_operator(const gdn_dims* dims, const void* k, const float* g, const float* beta, const void* v,
                       const int32_t* cu_seqlens, float* T_out, float* Slocal_out, void* stream) {
  g_last_error.clear();
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  int rc = check_token_dims(dims);
  if (rc) return rc;
  if (dims->n_seqs == 0) return GDN_OK;
  if (!cu_seqlens && dims->n_seqs != 1) return fail(GDN_ERR_ARG, "cu_seqlens may be NULL only for one chunk");
  if (!T_out || !Slocal_out) return fail(GDN_ERR_ARG, "T_out and Slocal_out are required");
  if (dims->total_tokens > 0 && (!k || !v || !g || !beta))
    return fail(GDN_ERR_ARG, "k, v, g and beta are required when total_tokens > 0");
  const void* p16[] = {k, v, T_out, Slocal_out};
  for (const void* p : p16)
    if (p && !aligned(p, 16)) return fail(GDN_ERR_ALIGN, "k, v, T_out and Slocal_out must be 16-byte aligned");
  if (!aligned(g, 4) || !aligned(beta, 4) || !aligned(cu_seqlens, 4))
    return fail(GDN_ERR_ALIGN, "g, beta and cu_seqlens must be 4-byte aligned");
  int* status = device_status_word();
  if (!status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");

  SimtParams p{};
  p.q = nullptr; p.k = k; p.v = v; p.g = g; p.beta = beta; p.cu = cu_seqlens; p.S0 = nullptr;
  p.O = nullptr; p.S_out = Slocal_out; p.T_out = T_out;
  p.n_seqs = dims->n_seqs; p.total_tokens = dims->total_tokens;
  p.h_k = dims->h_k; p.h_v = dims->h_v; p.d_k = dims->d_k; p.d_v = dims->d_v;
  p.augmented = 1; p.l2norm = (dims->flags & GDN_QK_L2NORM) ? 1 : 0;
  p.write_O = 0; p.scale = 1.f; p.status = status;
  p.scalar_decay = (dims->flags & GDN_SCALAR_DECAY) ? 1 : 0;
  // Two passes: the chunk-shared quantities once per (chunk, v-head) into pool scratch, then the
  // row slices of the augmented state [S; P] read them.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = simt_records_bytes(p.n_seqs, p.total_tokens, p.h_v);
  cudaMemPool_t pool = nullptr;
  int prc = scratch_pool(&pool);
  if (prc) return prc;
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, st);
  if (e != cudaSuccess) return fail(GDN_ERR_NOMEM, "scratch of %zu bytes: %s", bytes, cudaGetErrorString(e));
  e = launch_replay_simt_two_pass(p, dims->dtype == GDN_BF16, ws, bytes, st);
  const cudaError_t ef = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, "gdn_chunk_operator launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch release");
  return GDN_OK;
}

int gdn_compose(const gdn_dims* dims, int32_t K, const float* const* T, const float* const* Slocal,
                const float* S_in, float* S_out, void* stream) {
  g_last_error.clear();
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  int rc = check_head_dims(dims);
  if (rc) return rc;
  if (K < 0 || K > kMaxCompose) return fail(GDN_ERR_ARG, "K=%d outside [0, %d]", K, kMaxCompose);
  if (!S_out) return fail(GDN_ERR_ARG, "S_out is required");
  if (K > 0 && (!T || !Slocal)) return fail(GDN_ERR_ARG, "T and Slocal arrays are required when K > 0");
  ComposeParams p{};
  for (int j = 0; j < K; ++j) {
    if (!T[j] || !Slocal[j]) return fail(GDN_ERR_ARG, "T[%d] or Slocal[%d] is NULL", j, j);
    if (!aligned(T[j], 16) || !aligned(Slocal[j], 16)) return fail(GDN_ERR_ALIGN, "T[%d]/Slocal[%d] not 16-byte aligned", j, j);
    if (T[j] == S_out || Slocal[j] == S_out) return fail(GDN_ERR_ARG, "S_out aliases an input");
    p.T[j] = T[j];
    p.Slocal[j] = Slocal[j];
  }
  if ((S_in && !aligned(S_in, 16)) || !aligned(S_out, 16)) return fail(GDN_ERR_ALIGN, "S_in/S_out not 16-byte aligned");
  if (S_in && S_in == S_out) return fail(GDN_ERR_ARG, "S_out aliases S_in");
  p.S_in = S_in; p.S_out = S_out; p.K = K; p.h = dims->h_v; p.d_k = dims->d_k; p.d_v = dims->d_v;
  p.status = device_status_word();
  if (!p.status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  p.wait_ns = take_wait_limit_ns();
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = compose_tc_supported(p) ? launch_compose_tc(p, st) : launch_compose_simt(p, st);
  if (e != cudaSuccess) return cuda_fail(e, "gdn_compose launch");
  return GDN_OK;
}

int gdn_get_status(void* stream) {
  g_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  int st = 0;
  e = cudaMemcpyFromSymbol(&st, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (st != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return fail(st, "device reported status %d", st);
  }
  return GDN_OK;
}

}  // extern "C"
