/*
 * cpattn.h -- C ABI of the zigzag context-parallel causal attention library
 * (libcpattn.so, sm_103a).
 *
 * The computation is the one described on the page "context-parallel-
 * multimodal" (xuesongtap.github.io), called "CP-VLM page" below:
 *
 *   - §1.1: the text of a sequence is cut into 2P chunks and simulated
 *     context-parallel rank r keeps the head-tail pair (r, 2P-r-1), gathered
 *     with index_select on the sequence dimension;
 *   - §1 and the page's Ring Attention reference: every rank's queries meet
 *     every rank's keys in ring order, and the per-step partial results are
 *     merged by log-sum-exp;
 *   - §4.1: an image-token prefix is replicated, unsplit, to every rank and
 *     every text query sees all of it;
 *   - §4.2: every rank obtains its own gradient of the prefix and these are
 *     summed (the AllReduce);
 *   - §5.3: packed samples are described by cu_seqlens.
 *
 * All P ranks are partitions of one sequence held in one GPU's memory: the
 * ring "send" is a read of another partition and the AllReduce is a
 * fixed-order sum on the device.  There are no collectives.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned device memory unless a parameter says "host".
 *    The library never allocates device memory; scratch lives in a caller-
 *    supplied workspace whose size the *_workspace_size functions return.
 *    (It keeps a few page-locked host staging buffers of its own for the
 *    work lists it uploads.)
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream).  Host arrays are read before the call
 *    returns.  Calls sharing one workspace must be ordered on one stream.
 *  - Layouts: q, k, v, out, dout, dq, dk, dv are [T][H][d] row-major in
 *    natural token order ("THD").  lse is [H][T] fp32, natural log of the
 *    softmax normaliser after the scale:
 *        lse[h][i] = log sum_{j visible} exp(scale * q_i . k_j).
 *  - cu_seqlens is n_seqs+1 ascending int32 on the HOST; sample i occupies
 *    tokens [cu[i], cu[i+1]) and is laid out [prefix (prefix_len tokens),
 *    text].  Each text length must be divisible by 2P.  The mask is causal
 *    within each sample over [prefix, text] and blocks across samples.
 *  - Every device pointer must be 16-byte aligned (CP_ERR_ALIGNMENT).
 *  - Errors: every call returns a cp_status_t; cp_last_error() gives a
 *    thread-local message for the last failing call of that thread.  A device
 *    wait that exceeds its bound (see cp_set_wait_limit) makes the kernel
 *    record the fact in the workspace and return early; cp_workspace_status()
 *    reports it as CP_ERR_TIMEOUT.
 *  - Bounds-checked build (libcpattn_checked.so, compiled with
 *    -DCPATTN_BOUNDS_CHECK): before every TMA load, TMA reduce and global
 *    store the tensor-core kernels test the row and head index against the
 *    tensor's extent; an index outside it is not accessed, the kernel records
 *    the site in the status word and stops, and cp_workspace_status() reports
 *    CP_ERR_BOUNDS.  The normal build compiles these tests away.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_VERSION 1

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum */
  CP_ERR_SHAPE = 2,       /* text length % 2P != 0, d not in {64,128}, ... */
  CP_ERR_DTYPE = 3,       /* dtype not supported by this entry point */
  CP_ERR_ALIGNMENT = 4,   /* a device pointer is not 16-byte aligned */
  CP_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
  CP_ERR_CUDA = 6,        /* a CUDA runtime call failed (message has details) */
  CP_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up */
  CP_ERR_UNSUPPORTED = 8, /* no kernel for this device / configuration */
  CP_ERR_BOUNDS = 9       /* bounds-checked build only: a kernel met an index
                             outside its tensor, skipped the access and returned */
} cp_status_t;

typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype_t;

/* Message for the last failing call made by this thread ("" if none). */
const char* cp_last_error(void);
/* Static name of a status code. */
const char* cp_status_string(cp_status_t s);
/* CPATTN_VERSION of the loaded library. */
int cp_version(void);

/*
 * cp_zigzag_index -- the zigzag gather table and its inverse.
 * CP-VLM page §1.1 (index = [cp_rank, 2*cp_size-cp_rank-1], index_select on
 * the sequence dimension), applied to each sample's text (§4.1 step 3, §5.3).
 *
 *   fwd_idx[k] (k < P*R, R = sum_i text_len_i / P): natural token index of
 *     permuted text row k.  Rows are rank-major; within a rank sample-major;
 *     within a sample chunk r (c_i rows) then chunk 2P-r-1 (c_i rows), where
 *     c_i = text_len_i / (2P).
 *   inv_idx[m] (m < sum_i text_len_i): permuted row of the m-th text token in
 *     natural order (prefix tokens are not counted).
 *
 * on_device = 0: fwd_idx / inv_idx are host arrays, filled before return
 * (stream unused).  on_device = 1: they are device arrays (16-byte aligned),
 * written asynchronously on `stream` by the device kernel that cp_attn_fwd
 * runs for its own gather table; the per-sample table travels in the kernel
 * parameters (one launch per 192 samples), so nothing is allocated or copied.
 * Either pointer may be NULL to skip that table.
 * Errors: CP_ERR_INVALID_ARG (n_seqs < 1, P < 1, prefix_len < 0, null
 * cu_seqlens), CP_ERR_SHAPE (a text length < 0 or not divisible by 2P).
 */
cp_status_t cp_zigzag_index(const int32_t* cu_seqlens_h, int n_seqs, int prefix_len, int P,
                            int32_t* fwd_idx, int32_t* inv_idx, int on_device, void* stream);

/*
 * cp_zigzag_gather / cp_zigzag_scatter -- the vectorised row permutation of
 * CP-VLM page §1.1 (index_select) and its inverse.  Rows are `row_bytes`
 * contiguous bytes (a multiple of 16); idx is a device int32 table of n_rows
 * entries.  gather: dst[k] = src[idx[k]].  scatter: dst[idx[k]] = src[k].
 * Bit-exact copies.  src/dst must not overlap.
 * Errors: CP_ERR_INVALID_ARG, CP_ERR_ALIGNMENT (pointers or row_bytes).
 */
cp_status_t cp_zigzag_gather(const void* src, void* dst, size_t row_bytes, const int32_t* idx,
                             int n_rows, void* stream);
cp_status_t cp_zigzag_scatter(const void* src, void* dst, size_t row_bytes, const int32_t* idx,
                              int n_rows, void* stream);

/*
 * cp_copy_rows -- strided row copy between host and device memory (either
 * direction, or device to device), asynchronous on `stream`: for r < rows,
 * width bytes from src + r * src_pitch to dst + r * dst_pitch.  Not part of
 * the method: it moves a range of heads of a [T][H][d] tensor (width =
 * heads x d x element size, pitch = H x d x element size) so that a host
 * caller can stream the heads of a large problem through the device in
 * chunks, copies of one chunk overlapping the kernels of another.  Host
 * memory must be page-locked for the copy to be asynchronous.
 * Errors: CP_ERR_INVALID_ARG (null pointer, width > a pitch), CP_ERR_CUDA.
 */
cp_status_t cp_copy_rows(void* dst, size_t dst_pitch, const void* src, size_t src_pitch,
                         size_t width, size_t rows, void* stream);

/*
 * cp_attn_fwd -- context-parallel causal attention forward.
 * CP-VLM page §1.1 (zigzag split), §1 (Ring Attention), §4.1 (replicated
 * prefix), §5.3 (cu_seqlens).
 *
 * The text rows of q, k, v are gathered into rank-local order (the split).
 * At ring step s = 0..P-1 every simulated rank r meets the KV of rank
 * (r-s) mod P (step 0: [replicated prefix, own chunks]), and the per-step
 * partial results are merged by log-sum-exp; out/lse are written in natural
 * order.  Prefix query rows attend causally to their own prefix once.  On the
 * tensor-core path one persistent kernel walks, per query tile, the KV tiles
 * of every ring step in ring order, so the merge is its online softmax and no
 * partial result leaves the chip.  CP_F32 (and CP_BF16 under
 * CPATTN_FWD_PER_STEP=1) launch one kernel per ring step that merges into an
 * fp32 running result in the workspace; the last contributing step writes
 * out/lse.
 *
 *   q, k, v    [T][H][d], dtype dt (CP_BF16: tensor-core path, fp32
 *              accumulation; CP_F32: fp32 CUDA-core path)
 *   T          cu_seqlens_h[n_seqs]
 *   d          64 or 128
 *   out        [T][H][d], dtype dt (bf16 rounds to nearest even)
 *   lse        [H][T] fp32
 *   out_lo     NULL, or (CP_BF16 only) [T][H][d] bf16: receives the rounding
 *              remainder o - out of the fp32 result o, so that out + out_lo
 *              carries o to about 16 bits.  Pass it to cp_attn_bwd.
 *   workspace  >= cp_attn_fwd_workspace_size(...) bytes, 256-byte aligned;
 *              the size depends on softmax_scale (below)
 *
 * Softmax scales above 0.25 (e.g. scale 1 on queries that carry 1/sqrt(d)
 * already) make dQ large enough that one bf16 rounding of the probabilities
 * shows in it.  There the CP_BF16 path runs the products that take a
 * probability-sized operand on f16 operands (three more mantissa bits): in
 * this call P V, with V replaced by a per-call f16 copy V * 2^-e whose
 * largest magnitude lies in [2^14, 2^15), e a power of two found on the
 * device (|e| <= 60); O is multiplied back by 2^e in fp32.  The scaling is
 * exact, so the copy loses nothing for values within 2^29 of the largest.
 * The workspace then also holds that copy (T x H_kv x d x 2 bytes).
 * Errors: CP_ERR_INVALID_ARG, CP_ERR_SHAPE, CP_ERR_DTYPE, CP_ERR_ALIGNMENT,
 * CP_ERR_WORKSPACE, CP_ERR_CUDA, CP_ERR_UNSUPPORTED (CP_BF16 on a device
 * without tcgen05).  T == 0 is a no-op returning CP_OK.
 */
size_t cp_attn_fwd_workspace_size(cp_dtype_t dt, int T, int H, int d,
                                  const int32_t* cu_seqlens_h, int n_seqs, int P,
                                  int prefix_len, float softmax_scale);
cp_status_t cp_attn_fwd(const void* q, const void* k, const void* v, cp_dtype_t dt, int T,
                        int H, int d, const int32_t* cu_seqlens_h, int n_seqs, int P,
                        int prefix_len, float softmax_scale, void* out, float* lse,
                        void* out_lo, void* workspace, size_t ws_bytes, void* stream);

/*
 * cp_attn_fwd_noalloc -- cp_attn_fwd for callers that cannot allocate device
 * memory.  The source pages have no counterpart to this entry point.
 *
 * Some callers are not allowed to allocate: a host framework that owns the
 * whole device memory pool and forbids allocations outside its own allocator,
 * or a deployment that runs inside a fixed memory budget reserved up front.
 * Such callers cannot provide the workspace cp_attn_fwd needs.  This entry
 * point takes the same arguments minus the workspace and uses a fixed scratch
 * array of 64 MiB compiled into the library instead (every GPU that loads the
 * library holds it until the process exits).  It calls no cudaMalloc,
 * cudaFree or other allocating routine; work lists are copied from ordinary
 * host memory.
 *
 *  - Capacity: for CP_BF16 the scratch holds the work lists of the all-steps
 *    forward (every ring step of a query tile in one launch, merged on chip),
 *    the zigzag table and the rank-local q/k/v: 3 x rows x H x d x 2 bytes,
 *    rows = text tokens.  At d = 128 that is 768 bytes per (text token, head),
 *    so about 85 000 (token, head) pairs, e.g. 8192 tokens with 10 heads.
 *    Above softmax scale 0.25 the f16 copy of v adds 2 x T x H x d bytes.
 *    CP_F32 merges its ring steps through an fp32 running result held in the
 *    scratch as well (about 1.6 KB per pair at d = 128).  Larger problems
 *    return CP_ERR_WORKSPACE with the number of bytes they would need.
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call shares the one array and leaves its contents behind; the
 *    status word is cleared at the start of each call and everything else is
 *    written before it is read.  Calls that overlap on the GPU (other streams,
 *    other host threads) race on the scratch: order them on one stream.
 *  - Results equal cp_attn_fwd's (same kernels and schedule).  The status
 *    word is the first thing in the scratch and is cleared at the start of
 *    each call: cp_workspace_status(NULL, stream) reads it (CP_ERR_TIMEOUT
 *    when a bounded device wait of the last call gave up).
 * Errors: as cp_attn_fwd, plus CP_ERR_WORKSPACE when the problem exceeds the
 * fixed scratch.
 */
cp_status_t cp_attn_fwd_noalloc(const void* q, const void* k, const void* v, cp_dtype_t dt,
                                int T, int H, int d, const int32_t* cu_seqlens_h, int n_seqs,
                                int P, int prefix_len, float softmax_scale, void* out,
                                float* lse, void* out_lo, void* stream);

/*
 * cp_lse_merge -- merge n_parts partial attention results over disjoint key
 * sets by log-sum-exp (the Ring Attention combination the CP-VLM page relies
 * on in §1 and §4.1 step 5):
 *     lse = log sum_p exp(lse_p),   out = sum_p exp(lse_p - lse) * out_p.
 * A part with lse = -inf contributes nothing; if every part is -inf the row
 * gets lse = -inf and out = 0.  The merged lse comes first (the largest
 * lse_p, then the sum of exp(lse_p - max)); out then sums the parts in index
 * order, each read once (16-byte loads when d is a multiple of 4).
 *
 *   part_out  [n_parts][rows][H][d] fp32       part_lse [n_parts][H][rows] fp32
 *   out       [rows][H][d], dtype out_dt       lse      [H][rows] fp32
 * Errors: CP_ERR_INVALID_ARG, CP_ERR_ALIGNMENT, CP_ERR_DTYPE, CP_ERR_CUDA.
 */
cp_status_t cp_lse_merge(int n_parts, const float* part_out, const float* part_lse, int rows,
                         int H, int d, void* out, cp_dtype_t out_dt, float* lse, void* stream);

/*
 * cp_attn_bwd -- backward of cp_attn_fwd.  CP-VLM page §4.2.
 *
 * Uses the final lse of the forward: D_i = dO_i . o_i, then for every ring
 * step the partial gradients of each rank's queries against the KV it met;
 * text dK/dV are accumulated for the rank that owns the KV (on chip over all
 * ring steps, in ring-step order, and written once).  At step 0 each
 * rank produces its own gradient of the replicated prefix K/V; these per-rank
 * gradients and the prefix queries' own term are summed -- the single-GPU
 * stand-in for the page's AllReduce.  With prefix_grad_per_rank (and on the
 * CP_F32 path) each term is kept in its own slot and a separate kernel sums
 * the slots in fixed order (ranks 0..P-1, then the prefix-query term).
 * Without it, the CP_BF16 path sums the terms on chip: one work item per
 * prefix key tile walks every rank's query runs in a fixed order and writes
 * the sum (no slot memory, no separate pass).
 *
 *   q, k, v, out, dout  [T][H][d], dtype dt;  lse [H][T] fp32 (from cp_attn_fwd)
 *   out_lo              NULL, or the remainder written by cp_attn_fwd: then
 *                       D_i = dO_i . (out_i + out_lo_i), which keeps the bf16
 *                       rounding of the stored output out of dQ and dK (it
 *                       matters when |dQ| is large, e.g. softmax scale 1)
 *   dq, dk, dv          [T][H][d] fp32 outputs (overwritten)
 *   prefix_grad_per_rank  NULL, or [2][P+1][n_seqs*prefix_len][H][d] fp32:
 *                       receives the per-rank prefix dK (slot 0) and dV
 *                       (slot 1) before the sum; index P = prefix-query term.
 *   workspace           >= cp_attn_bwd_workspace_size(...) bytes; above
 *                       softmax scale 0.25 it also holds f16 copies of q and k
 *                       (scaled as V in cp_attn_fwd): the products S = Q K^T,
 *                       dQ = dS K and dK = dS^T Q then run on f16 operands,
 *                       dS rounded to f16 after a power-of-two scaling that
 *                       bounds it by 2^15 (from max |v| and max |dout|)
 * Errors: as cp_attn_fwd.
 */
size_t cp_attn_bwd_workspace_size(cp_dtype_t dt, int T, int H, int d,
                                  const int32_t* cu_seqlens_h, int n_seqs, int P,
                                  int prefix_len, float softmax_scale);
cp_status_t cp_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const void* out_lo, const float* lse, const void* dout, cp_dtype_t dt,
                        int T, int H, int d,
                        const int32_t* cu_seqlens_h, int n_seqs, int P, int prefix_len,
                        float softmax_scale, float* dq, float* dk, float* dv,
                        float* prefix_grad_per_rank, void* workspace, size_t ws_bytes,
                        void* stream);

/*
 * cp_attn_fwd_gqa / cp_attn_bwd_gqa -- cp_attn_fwd / cp_attn_bwd with grouped
 * KV heads (grouped-query attention; H_kv = 1 is multi-query attention).
 * The pages do not define this variant: every model they describe has one KV
 * head per query head.  It is the layout of models that keep fewer KV heads,
 * read this way: query head h attends with KV head h / G, G = H / H_kv (runs
 * of G consecutive query heads share a KV head).  With H_kv == H these calls
 * are exactly cp_attn_fwd / cp_attn_bwd.
 *
 *   q, out, dout, dq    [T][H][d]          lse [H][T]
 *   k, v, dk, dv        [T][H_kv][d]       (dk, dv sum the G query heads'
 *                                           contributions of each KV head)
 *   prefix_grad_per_rank  NULL or [2][P+1][n_seqs*prefix_len][H_kv][d] fp32
 *   workspace           >= cp_attn_{fwd,bwd}_workspace_size_gqa(...) bytes
 * Every other argument, the ring-step order, the merge and the prefix sum
 * are those of cp_attn_fwd / cp_attn_bwd.
 * Errors: as cp_attn_fwd / cp_attn_bwd, plus CP_ERR_SHAPE when H_kv < 1 or H
 * is not a multiple of H_kv.
 */
size_t cp_attn_fwd_workspace_size_gqa(cp_dtype_t dt, int T, int H, int H_kv, int d,
                                      const int32_t* cu_seqlens_h, int n_seqs, int P,
                                      int prefix_len, float softmax_scale);
cp_status_t cp_attn_fwd_gqa(const void* q, const void* k, const void* v, cp_dtype_t dt, int T,
                            int H, int H_kv, int d, const int32_t* cu_seqlens_h, int n_seqs,
                            int P, int prefix_len, float softmax_scale, void* out, float* lse,
                            void* out_lo, void* workspace, size_t ws_bytes, void* stream);
size_t cp_attn_bwd_workspace_size_gqa(cp_dtype_t dt, int T, int H, int H_kv, int d,
                                      const int32_t* cu_seqlens_h, int n_seqs, int P,
                                      int prefix_len, float softmax_scale);
cp_status_t cp_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* out,
                            const void* out_lo, const float* lse, const void* dout,
                            cp_dtype_t dt, int T, int H, int H_kv, int d,
                            const int32_t* cu_seqlens_h, int n_seqs, int P, int prefix_len,
                            float softmax_scale, float* dq, float* dk, float* dv,
                            float* prefix_grad_per_rank, void* workspace, size_t ws_bytes,
                            void* stream);

/*
 * cp_workspace_status -- synchronise `stream` and report whether a kernel of
 * the last cp_attn_fwd / cp_attn_bwd call that used `workspace` gave up on a
 * bounded device wait (CP_ERR_TIMEOUT), met an index outside a tensor
 * (CP_ERR_BOUNDS, bounds-checked build only) or CP_OK.  workspace = NULL: the same
 * for the last cp_attn_fwd_noalloc call on the current device (its fixed
 * scratch holds the status word).
 */
cp_status_t cp_workspace_status(const void* workspace, void* stream);

/*
 * cp_plan_pairs -- host-only introspection of the ring-step work lists: for
 * every step s < P, the number of visible (query, key) pairs the forward and
 * the backward work lists cover (prefix-query pairs are part of step 0) and
 * the number of work items.  Forward figures are those of the 256-query items
 * of the tensor-core kernel; the 128-query items of the CUDA-core kernel are
 * checked to cover the same pairs, and the all-steps items of the default
 * tensor-core forward (every ring step of one query tile in one item) and
 * backward (every ring step of one key tile in one item, one item per key
 * tile and prefix slot) to cover their sums.  Any output may be NULL.  Needs
 * no GPU.
 * Errors: CP_ERR_INVALID_ARG, CP_ERR_SHAPE, CP_ERR_UNSUPPORTED (the work
 * lists disagree: an internal error).
 */
cp_status_t cp_plan_pairs(const int32_t* cu_seqlens_h, int n_seqs, int prefix_len, int P,
                          int64_t* fwd_pairs, int64_t* bwd_pairs, int64_t* fwd_items,
                          int64_t* bwd_items);

/*
 * cp_plan_unit_lists -- host-only view of how the default tensor-core forward
 * (all ring steps in one persistent launch) hands its units to `grid` CTAs.
 * An item is one 256-query tile with the key runs of every ring step (CP-VLM
 * page §1 ring order, §1.1 zigzag chunks, §4.1 prefix); a unit is an
 * (item, query head) pair, numbered item + n_items * head.
 *
 *   n_items   out: number of items (may be NULL)
 *   tiles     [n_items] or NULL: KV tiles each item visits (its cost)
 *   units     [n_items * H] or NULL: the units, CTA by CTA
 *   cta_off   [grid + 1] or NULL: CTA b walks units[cta_off[b] .. cta_off[b+1])
 *
 * Call once with NULL arrays to learn n_items.  The library applies these
 * lists when a launch has at least four units per SM, with grid = the SM
 * count; below that it launches one CTA per unit.  Needs no GPU.
 * Errors: CP_ERR_INVALID_ARG (H < 1, grid < 1, bad counts), CP_ERR_SHAPE.
 */
cp_status_t cp_plan_unit_lists(const int32_t* cu_seqlens_h, int n_seqs, int prefix_len, int P,
                               int H, int grid, int64_t* n_items, int32_t* tiles,
                               int32_t* units, int32_t* cta_off);

/*
 * cp_profile_begin / cp_profile_end -- instrumentation: between the two calls
 * the library records a pair of CUDA events on the launching stream around
 * every kernel it launches (any thread).  The tensor-core forward is one
 * launch covering all ring steps; with CPATTN_FWD_PER_STEP=1 in the
 * environment it is P ring-step launches, which overlap one another's tails
 * and share one pair that counts as P launches.  The tensor-core backward is
 * one launch covering all ring steps.  Above softmax scale 0.25 the f16
 * operand copies are made inside the gather (forward) and preprocess
 * (backward) pairs, which then count 3 launches each.  cp_profile_end
 * synchronises those events and returns, per
 * kernel kind, the summed milliseconds and the launch count in ms[8] /
 * launches[8] (either may be NULL):
 *   0 zigzag index   1 zigzag gather   2 tensor-core forward (ring steps)
 *   3 backward preprocess   4 tensor-core backward (ring steps)
 *   5 prefix-gradient sum   6 CUDA-core forward step   7 CUDA-core backward step
 * Errors: CP_ERR_CUDA.
 */
void cp_profile_begin(void);
cp_status_t cp_profile_end(double* ms, int64_t* launches);

/*
 * cp_set_wait_limit -- bound, in polling rounds, for every device-side wait of
 * the tensor-core kernels launched afterwards by any thread (<= 0 restores
 * the default, about a second of waiting).  A test hook for the timeout path.
 */
void cp_set_wait_limit(long long rounds);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
