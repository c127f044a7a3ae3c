// Kernel launchers (device code lives in the *.cu files of this folder).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "plan.h"

namespace cpattn {

// Device error word kept at the start of every workspace.
struct DevStatus {
  int32_t timeout;     // 1: a bounded wait gave up; 3: an index check failed
  int32_t where;       // site code of the first failure
  int32_t pad[62];
};
constexpr size_t kStatusBytes = 256;

// ---- memory kernels (kmem.cu) ----------------------------------------------
cudaError_t launch_gather_rows(const void* const* src, void* const* dst, int n_tensors,
                               size_t row_bytes, const int32_t* idx, int n_rows, bool scatter,
                               cudaStream_t st);
// Zigzag tables on the device.  `samples_host` is a HOST array [n_seqs][4]
// (first text token, chunk length c, rank-local offset, text ordinal of the
// first text token); it is passed to the kernel by value, kZigzagBatch
// samples per launch, so the call needs no device copy of it.
constexpr int kZigzagBatch = 192;
struct ZigzagBatch {
  int n, P;
  long long R;          // rank-local rows per rank (all samples)
  long long loc0;       // rank-local row of the batch's first sample
  long long span;       // rank-local rows the batch covers on each rank
  int32_t smp[kZigzagBatch][4];
};
cudaError_t launch_zigzag_index(const int32_t* samples_host, int n_seqs, int P, int64_t R,
                                int32_t* fwd_idx, int32_t* inv_idx, cudaStream_t st);
cudaError_t launch_lse_merge(int n_parts, const float* part_out, const float* part_lse, int rows,
                             int H, int d, void* out, bool out_bf16, float* lse, cudaStream_t st);
// D[h*pitch + t] = sum_e dO[t][h][e] * O[t][h][e];  lse2[h*pitch + t] = lse[h][t] * log2(e)
// (out_lo nullable, bf16 only: D uses out + out_lo)
cudaError_t launch_bwd_preprocess(const void* out, const void* out_lo, const void* dout, bool bf16,
                                  const float* lse, int T, int H, int d, float* D, float* lse2,
                                  int64_t pitch, cudaStream_t st);
// dk/dv prefix rows = sum over slots 0..P of the per-rank prefix gradients
cudaError_t launch_prefix_reduce(const float* slots_k, const float* slots_v, int n_slots,
                                 const int32_t* cu_dev, int n_seqs, int N, int H, int d,
                                 float* dk, float* dv, cudaStream_t st);

// ---- fp32 inputs: CUDA-core attention (attn_simt.cu) -------------------------
struct SimtFwdArgs {
  const void* q_text; const void* k_text; const void* v_text;  // SRC_TEXT tensors
  const void* q_nat; const void* k_nat; const void* v_nat;     // SRC_NAT tensors
  const FwdItem* items; int n_items;
  int H, d; float scale;
  int Hkv;                                          // KV heads (query head h reads h / (H / Hkv))
  float* o_run; float* lse_run; int64_t run_rows;   // [H][run_rows][d], [H][run_rows]
  void* out; float* lse; int64_t T;                 // natural order
};
cudaError_t launch_simt_fwd(const SimtFwdArgs& a, cudaStream_t st);

struct SimtBwdArgs {
  const void* q; const void* k; const void* v; const void* dout;  // natural order
  const float* D; const float* lse2; int64_t pitch;               // [H][pitch]
  int H, d; float scale; int64_t T;
  int Hkv;                                 // KV heads; dK/dV sum each group's query heads
  const FwdItem* q_items; int n_q_items;   // dQ pass (natural-order forward plan)
  const BwdItem* k_items; int n_k_items;   // dK/dV pass
  float* dq; float* dk; float* dv;
  float* pre_k; float* pre_v; int64_t pre_rows;   // [P+1][pre_rows][Hkv][d]
};
cudaError_t launch_simt_bwd_dq(const SimtBwdArgs& a, cudaStream_t st);
cudaError_t launch_simt_bwd_dkdv(const SimtBwdArgs& a, cudaStream_t st);

}  // namespace cpattn
