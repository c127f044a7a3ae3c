// Attention backward over all ring steps in one launch, on 5th-generation
// tensor cores (sm_103a), with 128-query tiles so that every product is a
// 128 x 128 (x D) MMA.
//
// One CTA owns one key tile (128 keys of one KV head) and walks, in ring-step
// order, the query runs that meet those keys over all ring steps, for every
// query head that reads this KV head (page "context-parallel-multimodal"
// §4.2: each rank differentiates its queries against the KV it saw; the KV
// owner receives dK/dV, here summed on chip over the steps and written once;
// the replicated prefix gets one gradient per rank: one item per slot when
// the per-rank terms are kept, else one item that walks every rank's queries
// and writes their sum).  Per 128-row query tile i, with the final lse:
//
//   S^T  = K Q^T          dP^T = V dO^T                          (TMEM)
//   P^T  = exp2(S^T * scale*log2e - lse2),  dS^T = P^T (dP^T - D)  (registers)
//   dV  += P^T dO   (P^T read from TMEM)   dK += dS^T Q            (TMEM, whole item)
//   dQ   = dS K     -> staged per warp in swizzled shared memory, added
//                      into fp32 dQ (scaled) by bulk tensor reduce-adds
//
// Tensor memory (512 columns):
//   D = 128: S^T [0,128) (P^T overwrites its columns [0,32) and [64,96)),
//            dP^T [128,256) (dQ overwrites it once read), dK [256,384),
//            dV [384,512);
//   D = 64:  S^T [0,128), dP^T [128,256), dK [256,320), dV [320,384),
//            dQ [384,448).
// Issue order per tile: dP_i, dV_i, S_{i+1}, dQ_i, dK_i.  The P part of the
// softmax work of tile i runs while dQ_{i-1}, dK_{i-1} and dP_i compute; the
// dS part while dV_i and S_{i+1} do; the dQ drain while dK_i does.  With
// D = 128, dP_{i+1} waits for the drain to have read dQ_i out of the dP^T
// columns.
//
// For softmax scales above kF16OperandScale the dQ values are large enough
// that one bf16 rounding of dS would dominate their error.  S^T, dQ and dK
// then run on f16 operands: the host-made copies Q * 2^-eQ and K * 2^-eK, and
// dS^T * 2^-eS rounded to f16 (three more mantissa bits than bf16); the
// factors are undone in fp32 (OpScales).  dP^T and dV keep bf16 V, dO and P^T.
//
// Warp roles (512 threads; TMEM lane quarter of warp w is w % 4):
//   warp 0       TMA producer: K, V once; Q and the lse2 / D rows per tile
//   warp 1       TMEM allocation; lane 0 issues every tcgen05.mma
//   warp 2       TMA producer: dO per tile
//   warp 3       idle
//   warps 4..11  P / dS (two warpgroups, 64 query columns each; thread = key
//                row), then the dK / dV epilogue
//   warps 12..15 dQ drain; thread = query row (TMEM lane of dQ)
// Registers: warpgroup 0 drops to 64 (the least that leaves its MMA and
// producer code without spills), the P / dS warpgroups rise to 136 and the
// drain warpgroup to 168 (128 * 64 + 256 * 136 + 128 * 168 <= 512 * 128), so a
// drain thread can hold its whole dQ row and free the TMEM at once.
#include <cuda_bf16.h>

#include <type_traits>

#include "check.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc.h"

namespace cpattn {

namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kBK = kBwdTileK;     // 128 keys
constexpr int kBQ = 128;           // queries per inner tile
constexpr int kQStages = 2;
constexpr int kLdRows = kBQ + 4;   // lse2 / D box: 128 rows plus alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128;
constexpr long long kDrainLimit = 1LL << 24;

template <int D>
struct Cols {
  static constexpr uint32_t kDK = 256;
  static constexpr uint32_t kDV = kDK + D;
  static constexpr uint32_t kDQ = D == 128 ? kColDP : kDV + D;   // D = 128: aliases dP^T
  static constexpr bool kAliased = D == 128;
};

template <int D>
struct Lay {
  static constexpr int kBox = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kTile = D / 64 * kBox;   // 128 rows x D bf16
  // dO is read only by dP_i and dV_i (adjacent products): with D = 128 one
  // buffer suffices and leaves room for the dQ staging
  static constexpr int kDOStages = D == 128 ? 1 : 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                     // [stage]
  static constexpr int kDO = kQ + kQStages * kTile;         // [stage]
  static constexpr int kDS = kDO + kDOStages * kTile;       // dS^T: 2 boxes [128 keys][64 q]
  static constexpr int kStg = kDS + 2 * kBox;
  static constexpr int kStgWarp = 32 * 128;                 // [32 rows][32 fp32], 128-byte swizzle
  static constexpr int kLd = kStg + 4 * kStgWarp;           // [stage] {lse2[132], D[132]}
  static constexpr int kLdBytes = 2 * kLdRows * 4;
  static constexpr int kLdStride = (kLdBytes + 127) / 128 * 128;
  static constexpr int kItem = kLd + kQStages * kLdStride;
  static constexpr int kInfo = kItem + 128;                 // [stage] TileInfo of the Q tile
  static constexpr int kBars = kInfo + kQStages * 32;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kStg % 1024 == 0, "swizzled staging must be 1024-byte aligned");
  static_assert(kLd % 16 == 0 && (kLdRows * 4) % 16 == 0, "16-byte lse2 / D loads");
};
static_assert(Lay<128>::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(Lay<64>::kAlloc <= 227 * 1024, "shared memory budget");

// What the P / dS warps need of a query tile, written by the Q producer
// beside the tile (published by the same barrier as the Q load).
struct TileInfo {
  int32_t tile_row;   // natural row of the tile's first query
  int32_t row_in;     // the same query's position inside its run
  int32_t causal, delta, len;   // the run's visibility rule and length
  int32_t pad[3];
};
static_assert(sizeof(TileInfo) == 32, "TileInfo layout");

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, p_full, dp_full, ds_full;
  uint64_t dq_full, dq_free;
  uint64_t dkv_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ int run_qtiles(const Seg& s) {
  const int start = s.causal && s.delta < 0 ? -s.delta : 0;
  const int n = s.len - start;
  return n > 0 ? (n + kBQ - 1) / kBQ : 0;
}
__device__ __forceinline__ int run_qstart(const Seg& s) {
  return s.causal && s.delta < 0 ? -s.delta : 0;
}

// Each role walks the item's query tiles in order: g advances by one, or
// wraps to 0 for the next query head.  The walk keeps its current run and
// the number of tiles before it, so finding the g-th tile (its run, the run's
// first query and the tile index inside the run) costs one run read.
struct TileWalk {
  int s = 0, base = 0;
};
__device__ __forceinline__ void tile_of(const Seg* runs, int nseg, int g, TileWalk& w, Seg& sg,
                                        int& q0, int& t) {
  if (g < w.base) {
    w.s = 0;
    w.base = 0;
  }
  sg = runs[w.s];
  int nt = run_qtiles(sg);
  while (g >= w.base + nt && w.s + 1 < nseg) {
    w.base += nt;
    sg = runs[++w.s];
    nt = run_qtiles(sg);
  }
  q0 = run_qstart(sg);
  t = g - w.base;
}

__device__ __forceinline__ void record_timeout(int32_t* status, volatile int* abort, int site) {
  if (atomicCAS(&status[0], 0, 1) == 0) status[1] = site;
  *abort = 1;
}

template <int D, bool kF16, bool kShared>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_q128_kernel(const __grid_constant__ TcBwdArgs a) {
  using L = Lay<D>;
  using C = Cols<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps shared-space (not generic) loads and stores
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_idx = blockIdx.x % a.n_items;
  // KV head hk; its query heads are hk*G .. hk*G+G-1.  Shared groups
  // (kv_split > 1): kv_split CTAs take Gs = G / kv_split consecutive query
  // heads each, and their partial dK / dV meet in global memory by
  // reduce-adds.
  const int hk = kShared ? blockIdx.x / a.n_items / a.kv_split : blockIdx.x / a.n_items;
  const int G = a.H / a.Hkv;
  const int Gs = kShared ? G / a.kv_split : G;   // query heads of this CTA
  const int hq0 = hk * G + (kShared ? blockIdx.x / a.n_items % a.kv_split * Gs : 0);
  BwdItem& it = *reinterpret_cast<BwdItem*>(smem + L::kItem);
  if (warp == 0)  // the work item, copied once into shared memory (128 bytes)
    reinterpret_cast<uint32_t*>(&it)[lane] =
        reinterpret_cast<const uint32_t*>(a.items + item_idx)[lane];
  volatile int* abort = &bars->abort;
  const long long lim = a.wait_limit;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->do_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);
    mbar_init(&bars->dkv_done, 1);
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

  // the item's query runs, in ring-step order, from the plan's run list
  const int nseg = it.nseg;
  const Seg* runs = a.runs + it.run0;
  int n_qt = 0;   // query tiles of one query head
  for (int s = 0; s < nseg; ++s) n_qt += run_qtiles(runs[s]);
  // Every role walks the same Gs * n_qt query tiles in the same order: query
  // head hq0 + j / n_qt, tile j % n_qt.  dK / dV of the KV head accumulate
  // over all of them, across every ring step, and are written once.
  // Concurrent CTAs are neighbouring key tiles that meet the same queries in
  // the same order, so the Q / dO tiles they load are shared through L2.
  const int n_all = Gs * n_qt;

  if (warp < 4) {
    setmaxnreg_dec<64>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer: K, V, Q, lse2 / D
      if (lane == 0) {
        int issued = 0;
        bool kv_issued = false;
        if (n_all > 0 && !(CP_IN_RANGE(it.k_row0, 0, a.T, a.status, 201) &&
                           CP_IN_RANGE(hk, 0, a.Hkv, a.status, 202))) {
          *abort = 1;
        } else if (n_all > 0) {
          mbar_expect_tx(&bars->kv_full, 2 * L::kTile);
          for (int b = 0; b < D / 64; ++b) {
            tma_load_3d(&a.tm_k, &bars->kv_full, smem + L::kK + b * L::kBox, b * 64, hk, it.k_row0);
            tma_load_3d(&a.tm_v, &bars->kv_full, smem + L::kV + b * L::kBox, b * 64, hk, it.k_row0);
          }
          kv_issued = true;
        }
        TileWalk walk;
        int jt = 0, hq = hq0;
        for (int j = 0; j < n_all; ++j, jt = jt + 1 == n_qt ? 0 : jt + 1, hq += jt == 0) {
          const int st = j % kQStages;
          if (*abort || (j >= kQStages &&
                         !mbar_wait(&bars->q_empty[st], ((j / kQStages) - 1) & 1, lim, abort))) {
            record_timeout(a.status, abort, 21);
            break;
          }
          Seg sg;
          int q0, t;
          tile_of(runs, nseg, jt, walk, sg, q0, t);
          const int grow = sg.row0 + q0 + t * kBQ;   // natural row of the tile's first query
          if (!CP_IN_RANGE(grow, 0, a.T, a.status, 203) || !CP_IN_RANGE(hq, 0, a.H, a.status, 204)) {
            *abort = 1;
            break;
          }
          TileInfo* info = reinterpret_cast<TileInfo*>(smem + L::kInfo) + st;
          info->tile_row = grow;
          info->row_in = q0 + t * kBQ;
          info->causal = sg.causal;
          info->delta = sg.delta;
          info->len = sg.len;
          mbar_expect_tx(&bars->q_full[st], L::kTile + L::kLdBytes);
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(&a.tm_q, &bars->q_full[st], smem + L::kQ + st * L::kTile + b * L::kBox,
                        b * 64, hq, grow);
          // the lse2 / D box starts at the row rounded down to 4 (16-byte TMA alignment)
          tma_load_3d(&a.tm_ld, &bars->q_full[st], smem + L::kLd + st * L::kLdStride, grow & ~3,
                      hq, 0);
          issued = j + 1;
        }
        // every load issued here must land before the CTA exits (normally the
        // consumers already waited for them and these waits return at once)
        int zero = 0;
        if (kv_issued) mbar_wait(&bars->kv_full, 0, kDrainLimit, &zero);
        for (int x = issued - kQStages; x < issued; ++x) {
          if (x < 0) continue;
          mbar_wait(&bars->q_full[x % kQStages], (x / kQStages) & 1, kDrainLimit, &zero);
        }
      }
    } else if (warp == 2) {
      // ---------------------------------------------------------- TMA producer: dO
      if (lane == 0) {
        constexpr int S = L::kDOStages;
        int issued = 0;
        TileWalk walk;
        int jt = 0, hq = hq0;
        for (int j = 0; j < n_all; ++j, jt = jt + 1 == n_qt ? 0 : jt + 1, hq += jt == 0) {
          const int st = j % S;
          if (*abort || (j >= S && !mbar_wait(&bars->do_empty[st], ((j / S) - 1) & 1, lim, abort))) {
            record_timeout(a.status, abort, 22);
            break;
          }
          Seg sg;
          int q0, t;
          tile_of(runs, nseg, jt, walk, sg, q0, t);
          const int grow = sg.row0 + q0 + t * kBQ;
          if (!CP_IN_RANGE(grow, 0, a.T, a.status, 205) || !CP_IN_RANGE(hq, 0, a.H, a.status, 206)) {
            *abort = 1;
            break;
          }
          mbar_expect_tx(&bars->do_full[st], L::kTile);
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(&a.tm_do, &bars->do_full[st], smem + L::kDO + st * L::kTile + b * L::kBox,
                        b * 64, hq, grow);
          issued = j + 1;
        }
        int zero = 0;
        for (int x = issued - S; x < issued; ++x) {
          if (x < 0) continue;
          mbar_wait(&bars->do_full[x % S], (x / S) & 1, kDrainLimit, &zero);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        // K-major A and B; B (Q, dO) MN-major; A (dS), B (K) MN-major.  S^T, dQ
        // and dK take f16 operands when kF16 (K, Q copies and dS^T all f16);
        // dP^T and dV always bf16 (V, dO, P^T)
        constexpr uint32_t idesc_s = kF16 ? idesc_f16(kBK, kBQ, 0, 0) : idesc_bf16(kBK, kBQ, 0, 0);
        constexpr uint32_t idesc_dp = idesc_bf16(kBK, kBQ, 0, 0);
        constexpr uint32_t idesc_dv = idesc_bf16(kBK, D, 0, 1);
        constexpr uint32_t idesc_dk = kF16 ? idesc_f16(kBK, D, 0, 1) : idesc_bf16(kBK, D, 0, 1);
        constexpr uint32_t idesc_dq = kF16 ? idesc_f16(kBQ, D, 1, 1) : idesc_bf16(kBQ, D, 1, 1);
        const uint32_t k_addr = smem_u32(smem + L::kK), v_addr = smem_u32(smem + L::kV);
        const uint32_t ds_addr = smem_u32(smem + L::kDS);
        // S^T (into the S columns) from K and Q stage st
        auto issue_s = [&](int st) {
          const uint32_t q_addr = smem_u32(smem + L::kQ + st * L::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {      // over head dim
            const uint32_t o = (kk / 4) * L::kBox + (kk % 4) * 32;
            mma_bf16(tmem + kColS, sdesc_sw128(k_addr + o, 16, 1024),
                     sdesc_sw128(q_addr + o, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full);
        };
        bool ok = true;
        if (n_all > 0) {
          ok = mbar_wait(&bars->kv_full, 0, lim, abort) && mbar_wait(&bars->q_full[0], 0, lim, abort);
          if (ok) {
            tc_fence_after();
            issue_s(0);
          }
        }
        for (int i = 0; ok && i < n_all; ++i) {
          const int st = i % kQStages, so = i % L::kDOStages;
          // ---- dP^T_i = V dO_i^T
          if (!mbar_wait(&bars->do_full[so], (i / L::kDOStages) & 1, lim, abort) ||
              (C::kAliased && i >= 1 && !mbar_wait(&bars->dq_free, (i - 1) & 1, lim, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t do_addr = smem_u32(smem + L::kDO + so * L::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk / 4) * L::kBox + (kk % 4) * 32;
            mma_bf16(tmem + kColDP, sdesc_sw128(v_addr + o, 16, 1024),
                     sdesc_sw128(do_addr + o, 16, 1024), idesc_dp, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->dp_full);
          // ---- dV += P^T_i dO_i, P^T from the S columns (query pairs per column)
          if (!mbar_wait(&bars->p_full, i & 1, lim, abort)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBQ / 16; ++kk) {    // over queries
            const uint32_t pa = tmem + kColS + (kk / 4) * 64 + (kk % 4) * 8;
            mma_bf16_ts(tmem + C::kDV, pa, sdesc_sw128(do_addr + kk * 16 * 128, L::kBox, 1024),
                        idesc_dv, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->do_empty[so]);
          // ---- S^T_{i+1} (overwrites P^T_i: issued after dV_i)
          if (i + 1 < n_all) {
            const int st1 = (i + 1) % kQStages;
            if (!mbar_wait(&bars->q_full[st1], ((i + 1) / kQStages) & 1, lim, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(st1);
          }
          // ---- dQ_i = dS_i K, then dK += dS^T_i Q_i
          if (!mbar_wait(&bars->ds_full, i & 1, lim, abort) ||
              (!C::kAliased && i >= 1 && !mbar_wait(&bars->dq_free, (i - 1) & 1, lim, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {    // over keys
            const uint64_t kb = sdesc_sw128(k_addr + kk * 16 * 128, L::kBox, 1024);
            mma_bf16(tmem + C::kDQ, sdesc_sw128(ds_addr + kk * 16 * 128, L::kBox, 1024), kb,
                     idesc_dq, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->dq_full);
          const uint32_t q_addr = smem_u32(smem + L::kQ + st * L::kTile);
#pragma unroll
          for (int kk = 0; kk < kBQ / 16; ++kk) {    // over queries
            mma_bf16(tmem + C::kDK,
                     sdesc_sw128(ds_addr + (kk / 4) * L::kBox + (kk % 4) * 32, 16, 1024),
                     sdesc_sw128(q_addr + kk * 16 * 128, L::kBox, 1024), idesc_dk,
                     (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->q_empty[st]);
        }
        if (ok && n_all > 0) mma_commit(&bars->dkv_done);
        if (!ok) {
          record_timeout(a.status, abort, 23);
          // nothing issued by this thread may still be running at exit
          mma_commit(&bars->drain);
          int zero = 0;
          mbar_wait(&bars->drain, 0, kDrainLimit, &zero);
        }
      }
    }
  } else if (warp >= 12) {
    setmaxnreg_inc<168>();
    // ------------------------------------------------------------ dQ drain
    // thread = query row wq * 32 + lane of the tile (TMEM lane of dQ).  The
    // whole row comes out of TMEM first (its columns are free again for the
    // next product at once); then the warp stages it 32 columns at a time in
    // its own swizzled buffer, and lane 0 adds each staged [32 rows][32
    // columns] block into dQ by a bulk tensor reduce-add (the reduction runs
    // in L2; rows past the run carry exact zeros, rows past T are clipped by
    // the tensor map).
    const int wq = warp & 3;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    // dQ = scale * (dS K); with f16 operands also undo the dS and K factors
    const float dq_mul = kF16 ? a.scale * a.op_scales->dq_mul : a.scale;
    uint8_t* stg = smem + L::kStg + wq * L::kStgWarp;
    uint8_t* my_row = stg + lane * 128;
    const int sw = lane & 7;
    bool ok = true;
    bool pending = false;
    TileWalk walk;
    int jt = 0, hq = hq0;
    for (int j = 0; ok && j < n_all; ++j, jt = jt + 1 == n_qt ? 0 : jt + 1, hq += jt == 0) {
      Seg sg;
      int q0, t;
      tile_of(runs, nseg, jt, walk, sg, q0, t);
      const int grow = sg.row0 + q0 + t * kBQ + wq * 32;   // natural row of this warp's first query
      if (!mbar_wait(&bars->dq_full, j & 1, lim, abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_off + C::kDQ + c * 32, r[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence32(r[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->dq_free);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        // the previous reduce of this warp must have read the buffer
        if (pending && lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 v = make_float4(__uint_as_float(r[c][4 * x]) * dq_mul,
                                       __uint_as_float(r[c][4 * x + 1]) * dq_mul,
                                       __uint_as_float(r[c][4 * x + 2]) * dq_mul,
                                       __uint_as_float(r[c][4 * x + 3]) * dq_mul);
          *reinterpret_cast<float4*>(my_row + ((x ^ sw) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && CP_IN_RANGE(grow - wq * 32, 0, a.T, a.status, 207) &&
            CP_IN_RANGE(hq, 0, a.H, a.status, 208)) {
          tma_reduce_add_3d(&a.tm_dq, stg, c * 32, hq, grow);
          bulk_commit();
        }
        pending = true;
      }
    }
    if (lane == 0) bulk_wait_all();   // every reduce-add finished before exit
    if (!ok) record_timeout(a.status, abort, 24);
  } else {
    setmaxnreg_inc<136>();
    // ------------------------------------------------------------ P / dS
    // Two warpgroups share every query tile: warpgroup g (warps 4+4g .. 7+4g)
    // computes P^T / dS^T for query columns [64g, 64g + 64) of its key rows.
    const int g = (warp - 4) >> 2;
    const int u = (warp & 3) * 32 + lane;        // key row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // S^T = (K16 Q16^T) * qk_mul and dS16 = dS * ds_inv with f16 operands
    const float sl2 = kF16 ? a.scale_log2 * a.op_scales->qk_mul : a.scale_log2;
    const float ds_inv = kF16 ? a.op_scales->ds_inv : 1.f;
    const bool key_ok = u < it.k_len;
    const int sw = u & 7;
    bool ok = true;
    for (int i = 0; ok && i < n_all; ++i) {
      const int st = i % kQStages;
      if (!mbar_wait(&bars->s_full, i & 1, lim, abort) ||
          !mbar_wait(&bars->q_full[st], (i / kQStages) & 1, lim, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the slot is rewritten only after this tile's dK product, which waits
      // for this warpgroup's dS
      const TileInfo ti = reinterpret_cast<const TileInfo*>(smem + L::kInfo)[st];
      uint32_t rs[2][32];
      tmem_ld32(tmem + lane_off + kColS + g * 64, rs[0]);
      tmem_ld32(tmem + lane_off + kColS + g * 64 + 32, rs[1]);
      tmem_ld_wait();
      reg_fence32(rs[0]);
      reg_fence32(rs[1]);
      const int tile_row = ti.tile_row;                     // natural row of the tile's first query
      const int row0 = ti.row_in + g * 64;                  // first query of this half (inside the run)
      const float* ld = reinterpret_cast<const float*>(smem + L::kLd + st * L::kLdStride) +
                        (tile_row & 3) + g * 64;
      // key u is visible to query row0 + x iff x < len - row0 and, for a causal
      // run, u <= row0 + x + delta
      const int first_vis = ti.causal ? u - ti.delta - row0 : 0;
      const int end_vis = key_ok ? ti.len - row0 : 0;
      const bool whole = __all_sync(0xffffffffu, first_vis <= 0 && end_vis >= 64);
      const bool vec = (tile_row & 3) == 0;
      // ---- P^T: probabilities of the 64 queries, computed in place over S and
      // kept in fp32 for dS; bf16 pairs into the first 32 of this warpgroup's
      // S columns
#pragma unroll
      for (int x = 0; x < 64; x += 4) {
        float l[4];
        if (vec) {
          const float4 l4 = *reinterpret_cast<const float4*>(ld + x);
          l[0] = l4.x; l[1] = l4.y; l[2] = l4.z; l[3] = l4.w;
        } else {
#pragma unroll
          for (int y = 0; y < 4; ++y) l[y] = ld[x + y];
        }
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          uint32_t& e = rs[(x + y) >> 5][(x + y) & 31];
          float pv = ex2(fmaf(__uint_as_float(e), sl2, -l[y]));
          if (!whole && (x + y < first_vis || x + y >= end_vis)) pv = 0.f;
          e = __float_as_uint(pv);
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x)
          pk[x] = pack_bf16x2(__uint_as_float(rs[x >> 4][(2 * x) & 31]),
                              __uint_as_float(rs[x >> 4][(2 * x + 1) & 31]));
        tmem_st32(tmem + lane_off + kColS + g * 64, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      // ---- dS^T = P^T (dP^T - D), bf16 into shared memory (row u of box g,
      // 128-byte swizzle), 32 queries at a time
      if (!mbar_wait(&bars->dp_full, i & 1, lim, abort)) { ok = false; break; }
      tc_fence_after();
      uint8_t* srow = smem + L::kDS + g * L::kBox + u * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t rd[32];
        tmem_ld32(tmem + lane_off + kColDP + g * 64 + h * 32, rd);
        tmem_ld_wait();
        reg_fence32(rd);
        uint32_t hk[16];
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          float dd[4];
          if (vec) {
            const float4 d4 = *reinterpret_cast<const float4*>(ld + kLdRows + h * 32 + x);
            dd[0] = d4.x; dd[1] = d4.y; dd[2] = d4.z; dd[3] = d4.w;
          } else {
#pragma unroll
            for (int y = 0; y < 4; ++y) dd[y] = ld[kLdRows + h * 32 + x + y];
          }
#pragma unroll
          for (int y = 0; y < 4; y += 2) {
            const float d0 = __uint_as_float(rs[h][x + y]) * (__uint_as_float(rd[x + y]) - dd[y]);
            const float d1 =
                __uint_as_float(rs[h][x + y + 1]) * (__uint_as_float(rd[x + y + 1]) - dd[y + 1]);
            if constexpr (kF16)
              hk[(x + y) / 2] = pack_f16x2(d0 * ds_inv, d1 * ds_inv);
            else
              hk[(x + y) / 2] = pack_bf16x2(d0, d1);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int off = ((h * 4 + c) ^ sw) << 4;
          *reinterpret_cast<uint4*>(srow + off) =
              make_uint4(hk[c * 4], hk[c * 4 + 1], hk[c * 4 + 2], hk[c * 4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full);
    }
    // ------------------------------------------------------------ dK / dV epilogue
    if (ok && n_all > 0 && !mbar_wait(&bars->dkv_done, 0, lim, abort)) ok = false;
    if (!ok) {
      record_timeout(a.status, abort, 25);
    } else {
      tc_fence_after();
      // warpgroup 0 writes dK (scaled), warpgroup 1 writes dV
      float* dst;
      bool row_ok = key_ok && CP_IN_RANGE(hk, 0, a.Hkv, a.status, 209);
      if (it.dk_mode == DK_TEXT) {
        row_ok = row_ok && CP_IN_RANGE(it.k_row0 + u, 0, a.T, a.status, 210);
        dst = (g == 0 ? a.dk : a.dv) + ((long long)(it.k_row0 + u) * a.Hkv + hk) * D;
      } else {
        row_ok = row_ok && CP_IN_RANGE(it.slot, 0, a.n_slots, a.status, 211) &&
                 CP_IN_RANGE(it.dk_row0 + u, 0, a.pre_rows, a.status, 212);
        const long long row = (long long)it.slot * a.pre_rows + it.dk_row0 + u;
        dst = (g == 0 ? a.pre_k : a.pre_v) + (row * a.Hkv + hk) * D;
      }
      const bool first = (it.flags & F_FIRST) != 0;
      const float mul = g == 0 ? (kF16 ? a.scale * a.op_scales->dk_mul : a.scale) : 1.f;
      const uint32_t col = g == 0 ? C::kDK : C::kDV;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (n_all > 0) {
          tmem_ld32(tmem + lane_off + col + c * 32, r);
          tmem_ld_wait();
          reg_fence32(r);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = 0u;
        }
        if (!row_ok) continue;
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          float4 v = make_float4(__uint_as_float(r[x]) * mul, __uint_as_float(r[x + 1]) * mul,
                                 __uint_as_float(r[x + 2]) * mul, __uint_as_float(r[x + 3]) * mul);
          float4* d4 = reinterpret_cast<float4*>(dst + c * 32 + x);
          if constexpr (kShared) {    // sub-CTAs of one group meet here (zeroed first)
            red_add_v4(d4, v);
            continue;
          }
          if (!first) {
            const float4 o = *d4;
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
          }
          *d4 = v;
        }
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

template <int D, bool kF16, bool kShared>
cudaError_t launch_q128(const TcBwdArgs& a, cudaStream_t st) {
  constexpr int smem = Lay<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_q128_kernel<D, kF16, kShared>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.n_items * a.Hkv * a.kv_split;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  tc_bwd_q128_kernel<D, kF16, kShared><<<(unsigned)blocks, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_bwd_q128(const TcBwdArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  if (a.runs == nullptr) return cudaErrorInvalidValue;   // all-steps items only
  if (a.kv_split < 1 || (a.H / a.Hkv) % a.kv_split != 0) return cudaErrorInvalidValue;
  if (a.f16 && a.op_scales == nullptr) return cudaErrorInvalidValue;
  const bool sh = a.kv_split > 1;
  if (a.d == 128) {
    if (a.f16) return sh ? launch_q128<128, true, true>(a, st) : launch_q128<128, true, false>(a, st);
    return sh ? launch_q128<128, false, true>(a, st) : launch_q128<128, false, false>(a, st);
  }
  if (a.d != 64) return cudaErrorNotSupported;
  if (a.f16) return sh ? launch_q128<64, true, true>(a, st) : launch_q128<64, true, false>(a, st);
  return sh ? launch_q128<64, false, true>(a, st) : launch_q128<64, false, false>(a, st);
}

}  // namespace cpattn
