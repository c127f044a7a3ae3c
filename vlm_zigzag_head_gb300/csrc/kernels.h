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

// ---- f16 operand copies (kmem.cu) ---------------------------------------------
// Statistics and power-of-two factors of the f16 operand copies that the
// tensor-core kernels use above softmax scale 0.25, computed on the device
// (workspace) before the attention kernel reads them.
struct OpScales {
  uint32_t amax[4];   // bit patterns of max |x| (non-negative floats order as integers):
                      // forward V; backward Q, K, V, dO.  Zeroed before each call.
  int32_t e[4];       // copy of tensor t = x * 2^-e[t]
  float v_mul;        // forward: O = (P V16) * v_mul
  float qk_mul;       // backward: S = (K16 Q16^T) * qk_mul
  float ds_inv;       // backward: dS16 = dS * ds_inv (|dS16| < 2^15)
  float dq_mul;       // backward: dQ = scale * (dS16 K16) * dq_mul
  float dk_mul;       // backward: dK = scale * (dS16^T Q16) * dk_mul
  float pad[3];
};
static_assert(sizeof(OpScales) == 64, "OpScales layout");
// max |x| of up to 4 bf16 tensors of n[t] elements (multiples of 8, 16-byte
// aligned) into sc->amax[t] (atomic max over the bit patterns; NaN counts as
// the largest, and then gives the factor 1).
cudaError_t launch_absmax_bf16(const void* const* src, const int64_t* n, int n_tensors,
                               OpScales* sc, cudaStream_t st);
// dst[t] = f16(src[t] * 2^-e_t) for up to 2 bf16 tensors of n[t] elements,
// with e_t chosen from sc->amax[t] so that the largest magnitude lies in
// [2^14, 2^15) (clamped to |e_t| <= 60: the copies are exact for every value
// whose scaled magnitude is at least 2^-14).  Also fills sc's factors:
// backward = false: tensor 0 is V (v_mul); backward = true: tensors 0, 1 are
// Q and K, sc->amax[2], [3] hold max |V|, max |dO|, and d is the head size
// (qk_mul, ds_inv, dq_mul, dk_mul; dS is bounded by 2 d max|V| max|dO|).
cudaError_t launch_to_f16_scaled(const void* const* src, void* const* dst, const int64_t* n,
                                 int n_tensors, OpScales* sc, bool backward, int d,
                                 cudaStream_t st);

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
