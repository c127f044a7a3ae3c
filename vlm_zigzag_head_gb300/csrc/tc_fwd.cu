// Ring-step attention forward on 5th-generation tensor cores (sm_103a).
//
// A unit is one work item for one head: up to 256 query rows, taken as two
// 128-row tiles A and B, against a list of key runs (page
// "context-parallel-multimodal": §1.1 zigzag chunks, §1 ring order, §4.1
// replicated prefix in step 0), with an online softmax over the KV tiles.
// Two modes:
//   all steps in one launch (runs != null): the item's runs are those of
//     every ring step in ring order, so the online softmax itself is the
//     log-sum-exp merge of the per-step partials, and the epilogue writes
//     bf16 out and lse in natural order;
//   one ring step per launch: the epilogue merges into the fp32 running
//     result (or makes the final write at the query chunk's last step).
// Both tiles share every K / V tile.  The kernel is persistent: a CTA walks
// its own list of units (dealt by the host so that every CTA gets an equal
// share of KV tiles), or units gridDim.x apart without a list, with its
// barrier phases and K / V stages continuing from one unit to the next.
//
// The two tiles ping-pong: the tensor core computes one tile's products while
// the other tile's softmax runs.  Issue order for KV tile j >= 1:
//   PV_A(j-1)  S_A(j)  PV_B(j-1)  S_B(j)
// (S_A(j) overwrites the TMEM that holds P_A(j-1), so PV_A(j-1) goes first).
//
// Warp roles (384 threads; TMEM lane quarter of warp w is w % 4):
//   warp 0       TMA producer of K
//   warp 1       TMEM allocation; lane 0 issues every tcgen05.mma
//   warp 2       TMA producer of V
//   warp 3       TMA producer of Q (both tiles of a unit)
//   warps 4..7   softmax + epilogue of tile A; thread = query row = TMEM lane
//   warps 8..11  softmax + epilogue of tile B
//
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256, 256 + D),
// O_B [384, 384 + D).  P (bf16 pairs, 64 columns) overwrites the first half of
// its S buffer and is the A operand of PV, read straight from TMEM.  For
// softmax scales above kF16OperandScale P is rounded to f16 instead and V is
// the host-made f16 copy V * 2^-e (PV on f16 operands, O multiplied by 2^e in
// the epilogue): the backward's D = dO . O then carries O to about 11 bits,
// which keeps large dQ rows (few visible keys, scale 1) inside the bf16
// tolerance.  Shared
// memory: Q_A, Q_B, two K and two V stages (128 x D each) in the 128-byte
// swizzled layout TMA writes, 1024-byte aligned.
#include <cuda_bf16.h>

#include "check.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc.h"

namespace cpattn {

namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kBM = 128;         // rows of one query tile
constexpr int kBN = kFwdTileK;   // 128 keys per KV tile
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
// TMEM columns of tile x's S buffer and O accumulator
__device__ __forceinline__ uint32_t col_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max may lag by 2^8
constexpr long long kDrainLimit = 1LL << 24;

template <int D>
struct Smem {
  static constexpr int kTile = kBM * D * 2;        // bytes of a 128 x D bf16 tile
  static constexpr int kBox = 128 * 128;           // one 128-row x 128-byte TMA box
  static constexpr int kQ = 0;                     // [tile A, tile B]
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBars = kV + kStages * kTile;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};
static_assert(Smem<128>::kAlloc <= 227 * 1024, "shared memory budget");

struct Bars {
  uint64_t q_full, q_empty;   // Q of the CTA's current unit landed / free again
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2];   // per tile: S(j) in TMEM
  uint64_t p_full[2];   // per tile: P(j) in TMEM (4 softmax warps)
  uint64_t o_done[2];   // per tile: PV(j) accumulated
  uint64_t o_free[2];   // per tile: the epilogue has read O (4 softmax warps)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Tiles of one key run visible to query rows 0 .. q_len-1 of the item.
__device__ __forceinline__ int run_tiles(const Seg& s, int q_len) {
  int vis = s.len;
  if (s.causal) {
    vis = q_len + s.delta;
    vis = vis < 0 ? 0 : (vis < s.len ? vis : s.len);
  }
  return (vis + kBN - 1) / kBN;
}

// Key run s of an item: held in the item (one ring step per launch), or in
// the run list of the all-steps launch, where the item's runs are the runs of
// every ring step in ring order.
__device__ __forceinline__ Seg item_seg(const TcFwdArgs& a, const FwdItem& it, int s) {
  return a.runs != nullptr ? a.runs[it.run_row0 + s] : it.seg[s];
}

// The units this CTA walks, in order: without a unit table, u = blockIdx.x,
// blockIdx.x + gridDim.x, ... < n_units; with one, the table entries
// cta_off[blockIdx.x] .. cta_off[blockIdx.x + 1] - 1, where the host gave
// every CTA an equal share of work.  unit_id maps a position to the unit,
// item + n_items * query head.
struct UnitRange {
  int begin, end, step;
};
__device__ __forceinline__ UnitRange cta_units(const TcFwdArgs& a) {
  if (a.units != nullptr) return {a.cta_off[blockIdx.x], a.cta_off[blockIdx.x + 1], 1};
  return {(int)blockIdx.x, a.n_items * a.H, (int)gridDim.x};
}
__device__ __forceinline__ int unit_id(const TcFwdArgs& a, int u) {
  return a.units != nullptr ? a.units[u] : u;
}

// KV tiles an item visits over all its key runs.
__device__ __forceinline__ int item_tiles(const TcFwdArgs& a, const FwdItem& it) {
  int n = 0;
  for (int s = 0; s < it.nseg; ++s) n += run_tiles(item_seg(a, it, s), it.q_len);
  return n;
}

__device__ __forceinline__ void record_timeout(int32_t* status, volatile int* abort, int site) {
  if (atomicCAS(&status[0], 0, 1) == 0) status[1] = site;
  *abort = 1;
}

template <int D, bool kF16P>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ TcFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps shared-space (not generic) loads and stores
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  using L = Smem<D>;
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Persistent CTA: every role walks the CTA's units (cta_units) in the same
  // order.  KV tiles are numbered across units, so stage indices and barrier
  // phases simply continue; so are the units that visit at least one tile
  // ("tiled units", whose Q is loaded and whose O lives in TMEM).
  const int G = a.H / a.Hkv;   // query heads per KV head (grouped-query attention)
  volatile int* abort = &bars->abort;
  const long long lim = a.wait_limit;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], 4);
      mbar_init(&bars->o_done[x], 1);
      mbar_init(&bars->o_free[x], 4);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // the next ring step's CTAs may take SMs as this step's CTAs finish; they
  // wait for this grid before their merge epilogue (griddep_wait below)
  griddep_launch_dependents();
  // 384 threads launch with 168 registers each; warpgroup 0 (TMA, MMA) drops
  // to 72 and the two softmax warpgroups rise to 216, enough to hold a whole
  // 128-column S row: 128 * 72 + 256 * 216 = 384 * 168


  if (warp < 4) {
  setmaxnreg_dec<72>();
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers of K, V
    if (lane == 0) {
      const bool is_k = warp == 0;
      int issued = 0;
      int j = 0;   // KV tile counter across units
      const UnitRange ur = cta_units(a);
      for (int u = ur.begin; u < ur.end && !*abort; u += ur.step) {
        const int uid = unit_id(a, u);
        if (!CP_IN_RANGE(uid, 0, (long long)a.n_items * a.H, a.status, 101)) { *abort = 1; break; }
        const FwdItem& it = a.items[uid % a.n_items];
        const int hk = (uid / a.n_items) / G;
        for (int s = 0; s < it.nseg && !*abort; ++s) {
          const Seg sg = item_seg(a, it, s);
          if (!CP_IN_RANGE(sg.row0, 0, sg.src == SRC_TEXT ? a.text_rows : a.T, a.status, 102) ||
              !CP_IN_RANGE(hk, 0, a.Hkv, a.status, 103)) {
            *abort = 1;
            break;
          }
          const CUtensorMap* m = is_k ? (sg.src == SRC_TEXT ? &a.tm_k_text : &a.tm_k_nat)
                                      : (sg.src == SRC_TEXT ? &a.tm_v_text : &a.tm_v_nat);
          const int nt = run_tiles(sg, it.q_len);
          for (int t = 0; t < nt; ++t, ++j) {
            const int st = j % kStages;
            uint64_t* empty = is_k ? &bars->k_empty[st] : &bars->v_empty[st];
            uint64_t* full = is_k ? &bars->k_full[st] : &bars->v_full[st];
            if (j >= kStages && !mbar_wait(empty, ((j / kStages) - 1) & 1, lim, abort)) {
              record_timeout(a.status, abort, is_k ? 1 : 2);
              break;
            }
            uint8_t* dst = smem + (is_k ? L::kK : L::kV) + st * L::kTile;
            mbar_expect_tx(full, L::kTile);
            for (int b = 0; b < D / 64; ++b)
              tma_load_3d(m, full, dst + b * L::kBox, b * 64, hk, sg.row0 + t * kBN);
            issued = j + 1;
          }
        }
      }
      // every load this producer issued must land before the CTA exits
      // (normally the MMA issuer already waited for them: these return at once)
      int zero = 0;
      for (int x = issued - kStages; x < issued; ++x) {
        if (x < 0) continue;
        const int st = x % kStages;
        uint64_t* full = is_k ? &bars->k_full[st] : &bars->v_full[st];
        mbar_wait(full, (x / kStages) & 1, kDrainLimit, &zero);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ TMA producer of Q
    // Q of tiled unit n + 1 loads once the products of unit n are done.
    if (lane == 0) {
      int n = 0;   // tiled units so far
      const UnitRange ur = cta_units(a);
      for (int u = ur.begin; u < ur.end && !*abort; u += ur.step) {
        const int uid = unit_id(a, u);
        const FwdItem& it = a.items[uid % a.n_items];
        if (item_tiles(a, it) == 0) continue;
        if (n > 0 && !mbar_wait(&bars->q_empty, (n - 1) & 1, lim, abort)) {
          record_timeout(a.status, abort, 6);
          break;
        }
        if (!CP_IN_RANGE(it.q_row0, 0, it.q_src == SRC_TEXT ? a.text_rows : a.T, a.status, 104) ||
            !CP_IN_RANGE(uid / a.n_items, 0, a.H, a.status, 105)) {
          *abort = 1;
          break;
        }
        const CUtensorMap* qm = it.q_src == SRC_TEXT ? &a.tm_q_text : &a.tm_q_nat;
        mbar_expect_tx(&bars->q_full, 2 * L::kTile);
        for (int x = 0; x < 2; ++x)
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(qm, &bars->q_full, smem + L::kQ + x * L::kTile + b * L::kBox, b * 64,
                        uid / a.n_items, it.q_row0 + x * kBM);
        ++n;
      }
      int zero = 0;
      if (n > 0) mbar_wait(&bars->q_full, (n - 1) & 1, kDrainLimit, &zero);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = kF16P ? idesc_f16(kBM, D, 0, 1) : idesc_bf16(kBM, D, 0, 1);
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      // S_x(j) = Q_x K_j^T into tile x's S buffer
      auto issue_s = [&](int x, int j) {
        const uint32_t k_addr = smem_u32(smem + L::kK + (j % kStages) * L::kTile);
        const uint32_t qx = q_addr + x * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * L::kBox + (kk % 4) * 32;
          mma_bf16(tmem + col_s(x), sdesc_sw128(qx + off, 16, 1024),
                   sdesc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[x]);
      };
      // O_x += P_x(j) V_j, P from TMEM (keys 16kk.. 16kk+15: columns 8kk .. 8kk+7);
      // `first`: the unit's first tile, which overwrites O (after the previous
      // unit's epilogue has read it: o_free of tiled unit n - 1)
      auto issue_pv = [&](int x, int j, bool first, int n) -> bool {
        const int st = j % kStages;
        if (!mbar_wait(&bars->p_full[x], j & 1, lim, abort)) return false;
        if (x == 0 && !mbar_wait(&bars->v_full[st], (j / kStages) & 1, lim, abort)) return false;
        if (first && n > 0 && !mbar_wait(&bars->o_free[x], (n - 1) & 1, lim, abort)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + L::kV + st * L::kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v_addr + kk * 16 * 128, L::kBox, 1024);
          mma_bf16_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8, bd, idesc_pv,
                      (!first || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->o_done[x]);
        if (x == 1) mma_commit(&bars->v_empty[st]);
        return true;
      };
      bool ok = true;
      int j = 0;   // KV tile counter across units
      int n = 0;   // tiled units so far
      const UnitRange ur = cta_units(a);
      for (int u = ur.begin; ok && u < ur.end; u += ur.step) {
        const int n_tiles = item_tiles(a, a.items[unit_id(a, u) % a.n_items]);
        if (n_tiles == 0) continue;
        if (!mbar_wait(&bars->q_full, n & 1, lim, abort)) { ok = false; break; }
        const int j0 = j;
        for (int jj = 0; jj < n_tiles; ++jj, ++j) {
          const int st = j % kStages;
          if (!mbar_wait(&bars->k_full[st], (j / kStages) & 1, lim, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (jj >= 1 && !issue_pv(0, j - 1, j - 1 == j0, n)) { ok = false; break; }
          issue_s(0, j);
          if (jj >= 1 && !issue_pv(1, j - 1, j - 1 == j0, n)) { ok = false; break; }
          issue_s(1, j);
          mma_commit(&bars->k_empty[st]);
        }
        if (!ok) break;
        // the unit's S products, the only readers of Q, are all issued: the
        // next unit's Q may load while the last PV products run
        mma_commit(&bars->q_empty);
        if (!(issue_pv(0, j - 1, j - 1 == j0, n) && issue_pv(1, j - 1, j - 1 == j0, n))) {
          ok = false;
          break;
        }
        ++n;
      }
      if (!ok) {
        record_timeout(a.status, abort, 4);
        // drain: nothing issued by this thread may still be running at exit
        mma_commit(&bars->drain);
        int zero = 0;
        mbar_wait(&bars->drain, 0, kDrainLimit, &zero);
      }
    }
  }
  } else {
    setmaxnreg_inc<216>();
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;             // tile: 0 = A, 1 = B
    const int t = (warp & 3) * 32 + lane;      // query row of the tile == TMEM lane
    const int tq = x * kBM + t;                // query row of the item
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_off + col_s(x);
    const float sl2 = a.scale_log2;
    const float vmul = kF16P ? a.op_scales->v_mul : 1.f;   // V = V16 * vmul
    bool ok = true;
    int j = 0;   // KV tile counter across units
    const UnitRange ur = cta_units(a);
    for (int u = ur.begin; ok && u < ur.end; u += ur.step) {
    const int uid = unit_id(a, u);
    const FwdItem& it = a.items[uid % a.n_items];
    const int h = uid / a.n_items;
    const int q_len = it.q_len;   // rows of the item (tile A: first 128, tile B: the rest)
    const int nseg = it.nseg;
    const int n_tiles = item_tiles(a, it);
    const int j0 = j;
    float m = -INFINITY;   // running max of scaled scores (log2 units), may lag
    float l = 0.f;
    for (int s = 0; ok && s < nseg; ++s) {
      const Seg sg = item_seg(a, it, s);
      const int nt = run_tiles(sg, q_len);
      // key u of the run is visible to this row iff u < lim_u
      const int lim_u = sg.causal ? min(sg.len, tq + sg.delta + 1) : sg.len;
      for (int tt = 0; tt < nt; ++tt, ++j) {
        if (!mbar_wait(&bars->s_full[x], j & 1, lim, abort)) { ok = false; break; }
        tc_fence_after();
        // the whole 128-column S row of this thread in registers: one TMEM
        // round trip per tile
        uint32_t r[kBN / 32][32];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_col + c * 32, r[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) reg_fence32(r[c]);
        // keys at or past `vis` (tile-relative) are masked for this row
        const int vis = lim_u - tt * kBN;
        const bool whole = __all_sync(0xffffffffu, vis >= kBN);
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
        if (whole) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(r[i / 32][i % 32]));
        } else {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            mp[i & 7] = fmaxf(mp[i & 7], i < vis ? __uint_as_float(r[i / 32][i % 32]) : -INFINITY);
        }
        // max of the raw scores, then to scaled log2 units (scale > 0)
        const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl2;
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold || (m == -INFINITY && m_new != -INFINITY);
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m - m_new) : 1.f;  // m = -inf -> 0
          if (need) {
            l *= alpha;
            m = m_new;
          }
          if (j > j0) {  // O holds PV of earlier tiles (complete: PV_x(j-1) precedes S_x(j))
            if (!mbar_wait(&bars->o_done[x], (j - 1) & 1, lim, abort)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              const uint32_t col = tmem + lane_off + col_o(x) + c * 32;
              tmem_ld32(col, o);
              tmem_ld_wait();
              reg_fence32(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(col, o);
            }
            tmem_st_wait();
          }
        }
        // probabilities, row sum, and P (bf16 pairs, or f16 pairs for the f16 PV
        // product) over S columns [0, 64)
        const float mu = m == -INFINITY ? 0.f : m;
        float sp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sp[i] = 0.f;
        uint32_t pk[2][32];
        if (whole) {
#pragma unroll
          for (int i = 0; i < kBN; i += 2) {
            const float p0 = ex2(fmaf(__uint_as_float(r[i / 32][i % 32]), sl2, -mu));
            const float p1 = ex2(fmaf(__uint_as_float(r[i / 32][i % 32 + 1]), sl2, -mu));
            sp[(i >> 1) & 7] += p0 + p1;
            pk[i / 64][(i / 2) % 32] = pack_op2<kF16P>(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kBN; i += 2) {
            float p0 = ex2(fmaf(__uint_as_float(r[i / 32][i % 32]), sl2, -mu));
            float p1 = ex2(fmaf(__uint_as_float(r[i / 32][i % 32 + 1]), sl2, -mu));
            if (i >= vis) p0 = 0.f;
            if (i + 1 >= vis) p1 = 0.f;
            sp[(i >> 1) & 7] += p0 + p1;
            pk[i / 64][(i / 2) % 32] = pack_op2<kF16P>(p0, p1);
          }
        }
        tmem_st32(s_col, pk[0]);
        tmem_st32(s_col + 32, pk[1]);
        l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[x]);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0 && !mbar_wait(&bars->o_done[x], (j - 1) & 1, lim, abort))
      ok = false;
    // the running result was written by the previous ring step: its grid must
    // be complete (a no-op unless launched as a programmatic dependent)
    griddep_wait();
    if (!ok) {
      record_timeout(a.status, abort, 5);
      break;
    }
    {
      tc_fence_after();
      bool valid = tq < q_len;
      if (valid && (it.flags & F_FINAL) &&
          !(CP_IN_RANGE(it.out_row0 + tq, 0, a.T, a.status, 106) &&
            CP_IN_RANGE(h, 0, a.H, a.status, 107)))
        valid = false;   // checked build: the row is skipped
      if (valid && it.run_row0 >= 0 && a.runs == nullptr &&
          !CP_IN_RANGE(it.run_row0 + tq, 0, a.run_rows, a.status, 108))
        valid = false;
      float lse_s = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      const float inv = l > 0.f ? vmul / l : 0.f;
      const int flags = it.flags;
      const long long rrow =
          it.run_row0 >= 0 && a.runs == nullptr ? (long long)h * a.run_rows + it.run_row0 + tq : 0;
      float ca = 0.f, cb = 1.f;
      if (valid && !(flags & F_FIRST)) {
        const float lr = a.lse_run[rrow];
        const float mm = fmaxf(lr, lse_s);
        if (mm != -INFINITY) {
          const float wa = expf(lr - mm), wb = expf(lse_s - mm), tot = wa + wb;
          ca = wa / tot;
          cb = wb / tot;
          lse_s = mm + logf(tot);
        }
      }
      const float* orun = a.o_run + rrow * D;
      float* orun_w = a.o_run + rrow * D;
      const long long out_off = ((long long)(it.out_row0 + tq) * a.H + h) * D;
      __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(a.out) + out_off;
      __nv_bfloat16* lop =
          a.out_lo ? reinterpret_cast<__nv_bfloat16*>(a.out_lo) + out_off : nullptr;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_off + col_o(x) + c * 32, r);
          tmem_ld_wait();
          reg_fence32(r);
        } else {   // no key visible: O was never written for this unit
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (!valid) continue;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]) * inv;
        if (!(flags & F_FIRST)) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 pr = *reinterpret_cast<const float4*>(orun + c * 32 + i);
            o[i] = ca * pr.x + cb * o[i];
            o[i + 1] = ca * pr.y + cb * o[i + 1];
            o[i + 2] = ca * pr.z + cb * o[i + 2];
            o[i + 3] = ca * pr.w + cb * o[i + 3];
          }
        }
        if (flags & F_FINAL) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(o[i], o[i + 1]);
            v.y = pack_bf16x2(o[i + 2], o[i + 3]);
            v.z = pack_bf16x2(o[i + 4], o[i + 5]);
            v.w = pack_bf16x2(o[i + 6], o[i + 7]);
            *reinterpret_cast<uint4*>(outp + c * 32 + i) = v;
            if (lop) {  // remainder o - bf16(o), itself rounded to bf16
              float lo[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                lo[e] = o[i + e] - __bfloat162float(__float2bfloat16_rn(o[i + e]));
              uint4 w;
              w.x = pack_bf16x2(lo[0], lo[1]);
              w.y = pack_bf16x2(lo[2], lo[3]);
              w.z = pack_bf16x2(lo[4], lo[5]);
              w.w = pack_bf16x2(lo[6], lo[7]);
              *reinterpret_cast<uint4*>(lop + c * 32 + i) = w;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(orun_w + c * 32 + i) =
                make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
      }
      if (valid) {
        if (flags & F_FINAL) a.lse[(long long)h * a.T + it.out_row0 + tq] = lse_s;
        else a.lse_run[rrow] = lse_s;
      }
    }
    if (n_tiles > 0) {   // O of this unit is read: the next unit's first PV may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[x]);
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kF16P>
cudaError_t launch_d(const TcFwdArgs& a, cudaStream_t st) {
  const int smem = Smem<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel<D, kF16P>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM walks units gridDim.x apart
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.n_items * a.H;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // with few units per SM (under 4), one CTA per unit: a static share of
  // units per CTA would leave some CTAs a whole unit behind the others
  const long long blocks = a.units != nullptr ? a.n_ctas : fwd_grid(units, sms);
  if (blocks < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_fwd_kernel<D, kF16P>, a);
}

}  // namespace

cudaError_t launch_tc_fwd(const TcFwdArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  if (a.f16_pv) {
    if (a.op_scales == nullptr) return cudaErrorInvalidValue;
    return a.d == 64 ? launch_d<64, true>(a, st) : launch_d<128, true>(a, st);
  }
  return a.d == 64 ? launch_d<64, false>(a, st) : launch_d<128, false>(a, st);
}

}  // namespace cpattn
