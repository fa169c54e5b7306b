// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;    // tokens per scan chunk
constexpr int kMaxHead = 128; // largest d_k / d_v

// Parameters of one replay (or chunk-operator) launch on the fp32 CUDA-core path.
struct SimtParams {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const int32_t* cu;  // nullptr: one sequence of total_tokens
  const float* S0;
  void* O;
  float* S_out;   // value rows: [n_seqs][h_v][d_v][d_k]
  float* T_out;   // chunk-operator mode: [n_seqs][h_v][d_k][d_k]
  int n_seqs, total_tokens, h_k, h_v, d_k, d_v;
  int augmented;  // 1: state carries d_k extra transition rows (chunk operator)
  int l2norm;
  int write_O;
  int scalar_decay;  // 1: scalar per-token transition (no rank-1 projection term)
  float scale;
  int* status;    // sticky device status word
  unsigned char* rec;  // optional per-(chunk, v-head) records of the chunk-shared quantities (scratch)
};

// fp32 record of the chunk-shared quantities of one (chunk, v-head), written by the fp32 path's
// prep kernel: M = (I + A)^{-1} [64][64] (row t, column s), P [64][64] (only when outputs are
// wanted), then per token t: gamma_t, exp(G_last - G_t), beta_t, rk_t (key norm factor), rq_t
// (query norm factor times scale).  Offsets in floats.
constexpr int REC_M = 0, REC_P = 4096, REC_GAM = 8192, REC_WEND = 8256, REC_BETA = 8320, REC_RK = 8384,
              REC_RQ = 8448, REC_FLOATS = 8512;

cudaError_t launch_replay_simt(const SimtParams& p, int bf16, cudaStream_t stream);
// Scratch bytes of the two-kernel CUDA-core path (chunk-parallel prep, then the row-slice scan).
size_t simt_records_bytes(int n_seqs, int total_tokens, int h_v);
// The same computation as launch_replay_simt, with the chunk-shared work (norms, gates, Gram,
// (I + A)^{-1}) done once per (chunk, v-head) by a prep kernel into `workspace` first.
cudaError_t launch_replay_simt_two_pass(SimtParams p, int bf16, void* workspace, size_t bytes, cudaStream_t stream);

// Tensor-core path (bf16 inputs, d_k = d_v = 128, total_tokens > 0): a chunk-parallel
// prep kernel writes per-(chunk, v-head) records into `workspace`, then the scan
// kernel walks each tail.  workspace_bytes must be >= replay_tc_workspace_bytes().
bool replay_tc_supported(const SimtParams& p);
size_t replay_tc_workspace_bytes(int n_seqs, int total_tokens, int h_v);
cudaError_t launch_replay_tc(const SimtParams& p, void* workspace, size_t workspace_bytes, cudaStream_t stream);
int replay_tc_rows(int n_seqs, int h_v);

constexpr int kMaxCompose = 256;  // largest K of one gdn_compose call

// Passed by value: the K device pointers travel in the kernel parameters.
struct ComposeParams {
  const float* T[kMaxCompose];
  const float* Slocal[kMaxCompose];
  const float* S_in;
  float* S_out;
  int* status;  // sticky device status word (bounded waits that give up report GDN_ERR_TIMEOUT)
  unsigned long long wait_ns;  // limit of each bounded wait (0: give up unless already complete)
  int K, h, d_k, d_v;
};

cudaError_t launch_compose_simt(const ComposeParams& p, cudaStream_t stream);
// Tensor-core composition (split tf32, fp32 accuracy) for d_k = d_v = 128 and K >= 1.
bool compose_tc_supported(const ComposeParams& p);
cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t stream);

// Tensor map of a 2D bf16 view [rows][cols] (cols contiguous) with boxes of 64 columns x
// box_rows rows, 128-byte swizzle (the tile layout the tensor-core operands use); false if the
// driver's encoder is unavailable or rejects the view.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// The same for a 2D fp32 view: boxes of 32 columns (128 bytes) x box_rows rows.
bool make_map_f32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Operator-form state-only scan (bf16 inputs, d_k = d_v = 128, 32-row slices) over the records
// of the tensor-core prep kernel written with the Z factor (see state_tc.cu).
struct StateParams {
  const int32_t* cu;
  const int32_t* order;  // tails longest first, or null
  const float* S0;
  const unsigned char* rec;
  float* S_out;
  int* status;
  int n_seqs, total_tokens, h_k, h_v;
};
cudaError_t launch_state_tc(const CUtensorMap& mk, const CUtensorMap& mv, const StateParams& sp, bool overlap_prep,
                            cudaStream_t stream);

// Tensor-core state-only scan of the fp32 path (d_k = d_v = 128, fp32 or bf16 inputs, no
// outputs), over the records already written into p.rec: the state (augmented or not) in
// 128-row slices, at fp32 accuracy.
bool chunkop_tc_supported(const SimtParams& p, int bf16);
cudaError_t launch_chunkop_tc(const SimtParams& p, int bf16, cudaStream_t stream);

// Sticky status word of the current device (device pointer).
int* device_status_word();

// Helpers of the allocation-free replay entry point (defined in gdn_api.cu).
int check_replay_args(const gdn_dims* dims, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const int32_t* cu_seqlens, const float* S0, void* O_out, float* S_out,
                      SimtParams* p, bool* nothing_to_do);
int report_error(int code, const char* message);
// The event set by gdn_set_stage_event on this thread (nullptr if none); clears it.
void* take_stage_event();
// The wait limit set by gdn_set_wait_limit_ns on this thread (else the 2 s default); clears it.
unsigned long long take_wait_limit_ns();

}  // namespace gdn
