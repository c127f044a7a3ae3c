// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace cpattn {

// Softmax scales above this make dQ = scale * dS K large enough that one bf16
// rounding of a probability-sized operand (P in the forward's PV product, dS
// in the backward's dQ product) shows in dQ; both kernels then carry that
// operand as a bf16 hi + lo pair.
constexpr float kPrecisionSplitScale = 0.25f;

// 3-D tensor map over a bf16 [rows][H][d] tensor, box {64, 1, rows_per_box},
// 128-byte swizzle.  Returns false (and a message) if encoding fails.
bool make_tmap_thd(CUtensorMap* map, const void* base, int64_t rows, int H, int d,
                   int rows_per_box, const char** err);
// 3-D tensor map over an fp32 [rows][H][d] tensor, box {d, 1, box_rows}, no
// swizzle (the dQ reduce-add target of the backward).
bool make_tmap_f32_thd(CUtensorMap* map, void* base, int64_t rows, int H, int d, int box_rows,
                       const char** err);
// 3-D tensor map over an fp32 [rows][H][d] tensor, box {32, 1, box_rows} with
// the 128-byte swizzle (the dQ reduce-add target of the 128-query backward).
bool make_tmap_f32_sw128(CUtensorMap* map, void* base, int64_t rows, int H, int d, int box_rows,
                         const char** err);
// 3-D tensor map over the fp32 planes [2][H][pitch] (lse2, D) of the backward
// preprocess, box {box_rows, 1, 2}; pitch must be a multiple of 4.
bool make_tmap_ld(CUtensorMap* map, const void* base, int64_t pitch, int H, int box_rows,
                  const char** err);

struct TcFwdArgs {
  CUtensorMap tm_q_text, tm_k_text, tm_v_text;  // rank-local (gathered) text rows
  CUtensorMap tm_q_nat, tm_k_nat, tm_v_nat;     // natural order (prefix rows)
  const FwdItem* items;
  const Seg* runs;            // non-null: all ring steps in one launch; item key runs are
                              // runs[run_row0 .. run_row0 + nseg) (no running result)
  const int32_t* units;       // nullable: CTA b walks units[cta_off[b] .. cta_off[b + 1]),
  const int32_t* cta_off;     // entries item + n_items * head (a permutation of all units)
  int n_ctas;                 // grid size when units != null (cta_off has n_ctas + 1 entries);
                              // null units: CTA b walks b, b + grid, ...  (grid chosen here)
  int n_items, H, d;
  int Hkv;                    // KV heads; query head h reads KV head h / (H / Hkv)
  float scale_log2;           // softmax scale * log2(e)
  int split_p;                // P enters PV as bf16 hi + lo (softmax scale > kPrecisionSplitScale)
  int pdl;                    // launched as a programmatic dependent of the previous ring step
                              // (64-query kernel; the 128-query kernel is one launch per call)
  float* o_run; float* lse_run; int64_t run_rows;
  void* out; float* lse; int64_t T;
  void* out_lo;               // nullable: bf16 remainder o - bf16(o)
  int32_t* status;            // DevStatus of the workspace
  long long wait_limit;
  int64_t text_rows;          // rows of the rank-local (gathered) tensors (index checks)
};
cudaError_t launch_tc_fwd(const TcFwdArgs& a, cudaStream_t st);

struct TcBwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // natural order
  CUtensorMap tm_ld;                     // [2][H][pitch] fp32: lse2, D
  CUtensorMap tm_dq;                     // dq fp32 [T][H][d], box {d, 1, 16}: reduce-add target
  const BwdItem* items;
  const Seg* runs;            // run list of an all-steps plan (128-query kernel); else unused
  int n_items, H, d;
  int Hkv;                    // KV heads; one CTA per (key tile, KV head) walks its H / Hkv query heads
  float scale, scale_log2;
  int64_t T;
  float* dq; float* dk; float* dv;
  float* pre_k; float* pre_v; int64_t pre_rows;
  int32_t* status;
  long long wait_limit;
  int kv_split;               // CTAs sharing one KV head's query heads (divides H / Hkv); > 1:
                              // dK / dV / prefix slots are reduce-added into zeroed memory
  int pdl;                    // launched as a programmatic dependent of the previous ring step
                              // (64-query kernel; the 128-query kernel is one launch per call)
  int n_slots;                // prefix-gradient slots (P + 1) behind pre_k / pre_v (index checks)
};
cudaError_t launch_tc_bwd(const TcBwdArgs& a, cudaStream_t st);

// The backward walks 128-query tiles (tc_bwd_q128.cu: one launch over the
// all-steps plan, every item a key tile with the query runs of all ring
// steps) except at head_dim 128
// with the dS precision split, whose second dS buffer does not fit in shared
// memory beside 128-query tiles; that case walks 64-query tiles (tc_bwd.cu).
// The tensor maps differ: Q / dO boxes of bwd_tile_q(...) rows, an lse2 / D
// box of bwd_tile_q(...) + 4 rows, and the dQ target as swizzled 32-column
// boxes of 32 rows (128-query tiles) or unswizzled d-column boxes of 16 rows.
inline bool bwd_uses_q128(int d, float scale) { return d == 64 || scale <= kPrecisionSplitScale; }
inline int bwd_tile_q(int d, float scale) { return bwd_uses_q128(d, scale) ? 128 : 64; }
cudaError_t launch_tc_bwd_q128(const TcBwdArgs& a, cudaStream_t st);

}  // namespace cpattn
