// Work lists of the ring steps (host planner <-> kernels).
//
// The zigzag split (page "context-parallel-multimodal", §1.1) gives simulated
// rank r the text chunks r and 2P-r-1 of every sample (§5.3: per sample).  At
// ring step s rank r meets the KV of rank j = (r - s) mod P; at step 0 its
// local KV is [replicated image prefix, own chunks] (§4.1 step 4).  Whether a
// query chunk cq sees a key chunk ck follows from the global causal mask:
// ck < cq -> every pair visible, ck == cq -> causal within the chunk,
// ck > cq -> nothing.  The planner turns this into per-tile work items; the
// kernels only walk runs of rows with an optional causal rule.
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

namespace cpattn {

constexpr int kFwdTileQ = 128;  // query rows of one forward work item (CUDA-core path)
constexpr int kFwdPairQ = 256;  // query rows of one tensor-core forward item (two 128-row tiles)
constexpr int kFwdTileK = 128;  // keys per forward KV tile
constexpr int kBwdTileK = 128;  // keys of one backward work item
constexpr int kBwdTileQ = 64;   // query rows per backward inner tile
constexpr int kMaxSeg = 3;
constexpr int kBwdMaxSeg = 2;   // query runs of a per-step backward item (two chunks of a rank)

enum : int32_t { SRC_TEXT = 0, SRC_NAT = 1 };        // rank-local text buffer / natural order
enum : int32_t { F_FIRST = 1, F_FINAL = 2 };         // forward merge epilogue modes
enum : int32_t { DK_TEXT = 0, DK_PREFIX_SLOT = 1 };  // backward dK/dV destination

// A run of `len` consecutive rows starting at `row0` of tensor `src`.
// causal != 0: key u of the key run is visible to query t of the query run
// iff u <= t + delta (positions inside the same chunk / prefix).
struct Seg {
  int32_t row0, len, src, causal, delta, pad0, pad1, pad2;
};

// Forward: one query tile (<= kFwdTileQ rows) against up to kMaxSeg key runs.
struct FwdItem {
  int32_t q_row0, q_len, q_src, nseg;
  int32_t run_row0;  // row of the fp32 running result (rank-local order), -1: none
  int32_t out_row0;  // natural row of the first query (final write)
  int32_t flags;     // F_FIRST | F_FINAL
  int32_t n_tiles;   // KV tiles visited (cost)
  Seg seg[kMaxSeg];
};

// Backward: one key tile (<= kBwdTileK rows, natural order) against query
// runs (natural order): up to kBwdMaxSeg inline (per-step plans), or nseg
// runs of the plan's run list from run0 on (all-steps plans).
struct BwdItem {
  int32_t k_row0, k_len, nseg, n_tiles;
  int32_t dk_mode;  // DK_TEXT: dk/dv natural rows k_row0..; DK_PREFIX_SLOT: slot buffer
  int32_t dk_row0;  // row inside the prefix slot buffer (DK_PREFIX_SLOT)
  int32_t slot;     // prefix slot: rank 0..P-1, or P for the prefix queries' own term
  int32_t flags;    // F_FIRST: overwrite the destination, else accumulate
  int32_t run0;     // all-steps plans: index of the first run in the run list; else -1
  int32_t pad[7];
  Seg seg[kBwdMaxSeg];
};

static_assert(sizeof(Seg) == 32, "Seg layout");
static_assert(sizeof(FwdItem) == 128, "FwdItem layout");
static_assert(sizeof(BwdItem) == 128, "BwdItem layout");

struct Problem {
  int T = 0, P = 0, N = 0, n_seqs = 0;   // T = cu[n_seqs]
  std::vector<int32_t> cu;     // n_seqs + 1
  std::vector<int32_t> c;      // chunk length per sample
  std::vector<int32_t> off;    // rank-local offset of each sample (sum of 2c before it)
  int64_t R = 0;               // rank-local text rows per rank
  int64_t text_rows = 0;       // P * R
};

// Validates shapes (T < 0: do not check cu_seqlens[n] against T); returns ""
// on success or a message.
std::string make_problem(const int32_t* cu_seqlens, int n_seqs, int prefix_len, int P, int T,
                         Problem* out);

// Zigzag tables (natural index of permuted row; permuted row of text ordinal).
void zigzag_tables(const Problem& pb, int32_t* fwd_idx, int32_t* inv_idx);

struct FwdPlan {
  std::vector<FwdItem> items;
  std::vector<int32_t> step_begin;  // P + 1 offsets into items
};
struct BwdPlan {
  std::vector<BwdItem> items;
  std::vector<int32_t> step_begin;
};

// All ring steps fused per query tile: each item lists, in ring-step order,
// every key run its query tile meets over steps 0..P-1 (the runs of the
// per-step items of the same tile, concatenated).  An online softmax over
// those runs is the log-sum-exp merge of the per-step partials, taken one KV
// tile at a time.  Items: nseg = number of runs, run_row0 = index of the first
// run in `runs`, flags = F_FIRST | F_FINAL (no fp32 running result).
struct FusedFwdPlan {
  std::vector<FwdItem> items;
  std::vector<Seg> runs;
};
void plan_forward_fused(const FwdPlan& per_step, int P, FusedFwdPlan* out);

// CTAs of a tensor-core forward launch over `units` (item, head) units: one
// per unit below four units per SM, else one persistent CTA per SM.
inline long long fwd_grid(long long units, int sms) { return units < 4LL * sms ? units : sms; }

// Unit lists of a persistent forward launch with `grid` CTAs: CTA b walks
// units[cta_off[b] .. cta_off[b + 1]), each entry item + n_items * head.
// Units are taken head by head, items heaviest first (the plan's order), and
// each goes to the CTA with the least work so far (n_tiles plus a fixed cost
// per unit), as a dynamic scheduler would hand them out.  Every CTA's total
// then stays within one unit of the mean, and at any moment the CTAs work on
// one or two heads, whose K / V stay in L2.  (A plain round robin over
// (item, head) can give a CTA a much heavier share when n_items and grid
// share a stride.)
void plan_unit_lists(const std::vector<FwdItem>& items, int H, int grid,
                     std::vector<int32_t>* units, std::vector<int32_t>* cta_off);

// text_perm = true: text rows address the rank-local (gathered) buffer;
// false: they address natural order (used by the fp32 dQ pass).  tile_q:
// query rows per item (kFwdTileQ, or kFwdPairQ for the tensor-core kernel,
// which splits an item into two 128-row tiles; a causal rule then holds for
// the second tile with delta + 128).
void plan_forward(const Problem& pb, bool text_perm, FwdPlan* plan, int tile_q = kFwdTileQ);
void plan_backward(const Problem& pb, BwdPlan* plan);

// All ring steps fused per key tile (the mirror of FusedFwdPlan): each item
// lists, in ring-step order, every query run its key tile meets over steps
// 0..P-1, so that dK / dV accumulate on chip across the steps and are written
// once (flags = F_FIRST).  Items: nseg runs from run0 in `runs`; n_tiles =
// query tiles of tile_q rows (the cost); heaviest first.
// merge_prefix_slots = false: a prefix key tile has one item per slot (rank
// 0..P-1, and P for the prefix queries), written to its slot for the
// fixed-order sum that follows.  true: the slots' runs join one item that
// writes the summed prefix dK / dV straight to its natural rows (DK_TEXT):
// the same sum, taken on chip in the item's run order.
struct FusedBwdPlan {
  std::vector<BwdItem> items;
  std::vector<Seg> runs;
};
void plan_backward_fused(const BwdPlan& per_step, int P, int tile_q, bool merge_prefix_slots,
                         FusedBwdPlan* out);

}  // namespace cpattn
