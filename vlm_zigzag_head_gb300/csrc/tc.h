// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "plan.h"

namespace cpattn {

// Softmax scales above this make dQ = scale * dS K large enough that one bf16
// rounding of a probability-sized operand (P in the forward's PV product, dS
// in the backward's dQ and dK products) shows in dQ.  Those products then run
// on f16 operands (three more mantissa bits): P and dS are rounded to f16, and
// the other operand is a per-call f16 copy of V (forward) or of Q and K
// (backward), scaled by a power of two so that its largest magnitude lies in
// [2^14, 2^15).  The scaling is exact; the factors are undone in fp32.
constexpr float kF16OperandScale = 0.25f;
inline bool uses_f16_operands(float scale) { return scale > kF16OperandScale; }

// 3-D tensor map over a 16-bit [rows][H][d] tensor (bf16, or f16 when f16 is
// set), box {64, 1, rows_per_box}, 128-byte swizzle.  Returns false (and a
// message) if encoding fails.
bool make_tmap_thd(CUtensorMap* map, const void* base, int64_t rows, int H, int d,
                   int rows_per_box, const char** err, bool f16 = false);
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
  int f16_pv;                 // PV on f16 operands: P and the scaled copy of V behind
                              // tm_v_*; O is multiplied by op_scales->v_mul
  const OpScales* op_scales;  // device; read when f16_pv
  int pdl;                    // launched as a programmatic dependent of the previous ring step
  float* o_run; float* lse_run; int64_t run_rows;
  void* out; float* lse; int64_t T;
  void* out_lo;               // nullable: bf16 remainder o - bf16(o)
  int32_t* status;            // DevStatus of the workspace
  long long wait_limit;
  int64_t text_rows;          // rows of the rank-local (gathered) tensors (index checks)
};
cudaError_t launch_tc_fwd(const TcFwdArgs& a, cudaStream_t st);

struct TcBwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // natural order (Q, K: the f16 copies when f16)
  CUtensorMap tm_ld;                     // [2][H][pitch] fp32: lse2, D
  CUtensorMap tm_dq;                     // dq fp32 [T][H][d], box {32, 1, 32}, 128-byte swizzle:
                                         // reduce-add target
  const BwdItem* items;
  const Seg* runs;            // run list of the all-steps plan: item i's query runs are
                              // runs[items[i].run0 .. + nseg)
  int f16;                    // S, dQ and dK on f16 operands (scaled Q, K copies; dS in f16)
  const OpScales* op_scales;  // device; read when f16
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
  int n_slots;                // prefix-gradient slots (P + 1) behind pre_k / pre_v (index checks)
};
// The backward (tc_bwd_q128.cu): one launch over the all-steps plan, every
// item a key tile with the query runs of all ring steps, in 128-query tiles.
cudaError_t launch_tc_bwd_q128(const TcBwdArgs& a, cudaStream_t st);

}  // namespace cpattn
