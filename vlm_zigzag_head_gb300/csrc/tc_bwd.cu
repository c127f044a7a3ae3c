// Ring-step attention backward on 5th-generation tensor cores (sm_103a), with
// 64-query tiles: the form taken at head_dim 128 when the softmax scale is
// above kPrecisionSplitScale, where dS enters dQ as a bf16 hi + lo pair and the
// second dS buffer does not fit in shared memory beside 128-query tiles (every
// other case runs tc_bwd_q128.cu).
//
// One CTA owns one key tile (128 keys of one KV head) of a ring step and walks
// the query runs that met those keys at that step, for every query head that
// reads this KV head (one head without grouped KV heads) (page
// "context-parallel-multimodal" §4.2: each rank differentiates its queries
// against the KV it saw; the KV owner receives dK/dV; the replicated prefix
// gets one gradient per rank).  Per 64-row query tile, with the final lse:
//
//   S^T  = K Q^T            dP^T = V dO^T                      (TMEM)
//   P^T  = exp2(S^T * scale*log2e - lse2),  dS^T = P^T (dP^T - D)   (registers)
//   dV  += P^T dO           dK  += dS^T Q                      (TMEM, whole item)
//   dQ^T = K^T dS^T  -> staged in shared memory, added into fp32 dQ (scaled)
//                       by bulk tensor reduce-adds
//
// dS^T enters the dQ product as two bf16 terms, hi = bf16(dS^T) and
// lo = bf16(dS^T - hi), accumulated in fp32: with a softmax scale of 1 the
// dQ values are large enough that one bf16 rounding of dS would dominate the
// error.  dK and dV use the single bf16 rounding of dS^T and P^T.
//
// Warp roles (512 threads; TMEM lane quarter of warp w is w % 4):
//   warp 0       TMA producer (K, V once; Q, dO and the lse2 / D rows per query
//                tile, 3 stages)
//   warp 1       TMEM allocation; lane 0 issues every tcgen05.mma
//   warp 2       idle
//   warp 3       lane 0 issues the dQ bulk reduce-adds of the drain
//   warps 4..11  P / dS computation (two warpgroups, 32 query columns each),
//                then the dK / dV epilogue; thread = key row
//   warps 12..15 dQ drain into shared-memory staging; thread = head-dim
//                index (TMEM lane of dQ^T)
//
// TMEM columns: S^T [0,64), dP^T [64,128), dQ^T ping-pong [128,192) and
// [192,256), dK [256,384), dV [384,512).
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
constexpr int kD = 128;            // head dim of this kernel
constexpr int kBK = kBwdTileK;     // 128 keys
constexpr int kBQ = kBwdTileQ;     // 64 queries per inner tile
constexpr int kStages = 3;        // Q / dO / (lse2, D) stages
constexpr int kLdRows = kBQ + 4;  // lse2 / D box: 64 rows plus alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 64, kColDQ0 = 128, kColDQ1 = 192, kColDK = 256,
                   kColDV = 384;
constexpr long long kDrainLimit = 1LL << 24;

template <bool kSplit>
struct Lay {
  static constexpr int kKVBox = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int kQBox = kBQ * 128;    // 64 rows x 128 bytes
  static constexpr int kLdBytes = 2 * kLdRows * 4;
  static constexpr int kNumStg = kSplit ? 1 : 2;          // dQ staging buffers
  static constexpr int kStgRows = 16;                     // query rows per dQ reduce-add
  static constexpr int kStgBytes = kStgRows * kD * 4;     // 8 KB
  static constexpr int kK = 0;
  static constexpr int kV = kK + 2 * kKVBox;
  static constexpr int kQ = kV + 2 * kKVBox;              // [stage][2 boxes]
  static constexpr int kDO = kQ + kStages * 2 * kQBox;
  static constexpr int kP = kDO + kStages * 2 * kQBox;     // 128 x 64 bf16
  static constexpr int kDS = kP + kKVBox;                 // bf16(dS^T)
  static constexpr int kDSL = kDS + kKVBox;               // bf16(dS^T - bf16(dS^T)), split only
  static constexpr int kStg = kDSL + (kSplit ? kKVBox : 0);  // [buf][16][128] fp32 dQ staging
  static constexpr int kLd = kStg + kNumStg * kStgBytes;  // [stage] {lse2[68], D[68]}
  static constexpr int kItem = kLd + kStages * 1024;
  static_assert(kLd % 16 == 0 && (kLdRows * 4) % 16 == 0, "16-byte lse2 / D loads");
  static constexpr int kBars = kItem + 128;
  static constexpr int kBytes = kBars + 512;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(Lay<true>::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(Lay<false>::kAlloc <= 227 * 1024, "shared memory budget");

struct Bars {
  uint64_t kv_full;
  uint64_t qdo_full[kStages], qdo_empty[kStages];
  uint64_t sdp_full, sdp_empty;
  uint64_t ps_full, ps_empty;
  uint64_t dq_full[2], dq_empty[2];
  uint64_t dkv_done;
  uint64_t stg_full[2], stg_free[2];   // dQ staging buffers (drain warps / elected thread)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int run_qtiles(const Seg& s) {
  const int start = s.causal && s.delta < 0 ? -s.delta : 0;
  const int n = s.len - start;
  return n > 0 ? (n + kBQ - 1) / kBQ : 0;
}
__device__ __forceinline__ int run_qstart(const Seg& s) {
  return s.causal && s.delta < 0 ? -s.delta : 0;
}

// The g-th query tile of the item: its run, the run's first query and the
// tile index inside the run.
__device__ __forceinline__ void tile_of(const BwdItem& it, int g, Seg& sg, int& q0, int& t) {
  for (int s = 0; s < it.nseg; ++s) {
    const int nt = run_qtiles(it.seg[s]);
    if (g < nt) {
      sg = it.seg[s];
      q0 = run_qstart(sg);
      t = g;
      return;
    }
    g -= nt;
  }
}

__device__ __forceinline__ void record_timeout(int32_t* status, volatile int* abort, int site) {
  if (atomicCAS(&status[0], 0, 1) == 0) status[1] = site;
  *abort = 1;
}

template <bool kSplit, bool kShared>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_kernel(const __grid_constant__ TcBwdArgs a) {
  using L = Lay<kSplit>;
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
  BwdItem& it = *reinterpret_cast<BwdItem*>(smem + L::kItem);
  if (warp == 0)  // the work item, copied once into shared memory (128 bytes)
    reinterpret_cast<uint32_t*>(&it)[lane] =
        reinterpret_cast<const uint32_t*>(a.items + item_idx)[lane];
  volatile int* abort = &bars->abort;
  const long long lim = a.wait_limit;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qdo_full[s], 1);
      mbar_init(&bars->qdo_empty[s], 1);
    }
    mbar_init(&bars->sdp_full, 1);
    mbar_init(&bars->sdp_empty, 8);
    mbar_init(&bars->ps_full, 8);
    mbar_init(&bars->ps_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->dq_full[b], 1);
      mbar_init(&bars->dq_empty[b], 4);
    }
    mbar_init(&bars->dkv_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->stg_full[b], 4);
      mbar_init(&bars->stg_free[b], 1);
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
  // wait for this grid before their dK / dV epilogue (griddep_wait below)
  griddep_launch_dependents();

  const int nseg = it.nseg;
  int n_qt = 0;   // query tiles of one query head
  for (int s = 0; s < nseg; ++s) n_qt += run_qtiles(it.seg[s]);
  // Every role walks the same Gs * n_qt query tiles in the same order: the
  // CTA's first query head + j / n_qt, tile j % n_qt.  dK / dV of the KV head accumulate
  // over all of them.  Concurrent CTAs are neighbouring key tiles that meet
  // the same queries in the same order, so the Q / dO tiles they load are
  // shared through L2 (a rotated order per CTA measured slower).
  const int n_all = Gs * n_qt;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int issued = 0;
    bool kv_issued = false;
    if (n_all > 0 && lane == 0 &&
        !(CP_IN_RANGE(it.k_row0, 0, a.T, a.status, 301) && CP_IN_RANGE(hk, 0, a.Hkv, a.status, 302)))
      *abort = 1;
    if (n_all > 0 && !*abort) {
      if (lane == 0) {
        mbar_expect_tx(&bars->kv_full, 4 * L::kKVBox);
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(&a.tm_k, &bars->kv_full, smem + L::kK + b * L::kKVBox, b * 64, hk, it.k_row0);
          tma_load_3d(&a.tm_v, &bars->kv_full, smem + L::kV + b * L::kKVBox, b * 64, hk, it.k_row0);
        }
      }
      kv_issued = true;
    }
    // decisions are taken by lane 0 and broadcast: the warp never diverges
    // around the __syncwarp below
    bool go = true;
    int jt = 0, hq = hk * G + (kShared ? blockIdx.x / a.n_items % a.kv_split * Gs : 0);
    for (int j = 0; go && j < n_all; ++j, jt = jt + 1 == n_qt ? 0 : jt + 1, hq += jt == 0) {
      {
        Seg sg;
        int q0, t;
        tile_of(it, jt, sg, q0, t);
        const int st = j % kStages;
        int w_ok = 1;
        if (lane == 0) {
          w_ok = !*abort && (j < kStages ||
                             mbar_wait(&bars->qdo_empty[st], ((j / kStages) - 1) & 1, lim, abort));
          if (!w_ok) record_timeout(a.status, abort, 11);
        }
        go = __shfl_sync(0xffffffffu, w_ok, 0) != 0;
        if (!go) break;
        // Q, dO (64 rows each) and the lse2 / D rows of the tile; the lse2 / D
        // box starts at the row rounded down to 4 (16-byte TMA alignment)
        const int row0 = q0 + t * kBQ;
        const int grow = sg.row0 + row0;
        int c_ok = 1;
        if (lane == 0)
          c_ok = CP_IN_RANGE(grow, 0, a.T, a.status, 303) && CP_IN_RANGE(hq, 0, a.H, a.status, 304);
        if (!__shfl_sync(0xffffffffu, c_ok, 0)) {
          if (lane == 0) *abort = 1;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(&bars->qdo_full[st], 4 * L::kQBox + L::kLdBytes);
          for (int b = 0; b < 2; ++b) {
            tma_load_3d(&a.tm_q, &bars->qdo_full[st], smem + L::kQ + (st * 2 + b) * L::kQBox,
                        b * 64, hq, grow);
            tma_load_3d(&a.tm_do, &bars->qdo_full[st], smem + L::kDO + (st * 2 + b) * L::kQBox,
                        b * 64, hq, grow);
          }
          tma_load_3d(&a.tm_ld, &bars->qdo_full[st], smem + L::kLd + st * 1024, grow & ~3, hq, 0);
        }
        issued = j + 1;
      }
    }
    // every load issued here must have landed before the CTA exits (normally
    // the consumers already waited for them and these waits return at once)
    if (lane == 0) {
      int zero = 0;
      if (kv_issued) mbar_wait(&bars->kv_full, 0, kDrainLimit, &zero);
      for (int x = issued - kStages; x < issued; ++x) {
        if (x < 0) continue;
        mbar_wait(&bars->qdo_full[x % kStages], (x / kStages) & 1, kDrainLimit, &zero);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_sdp = idesc_bf16(kBK, kBQ, 0, 0);   // K-major A and B
      constexpr uint32_t idesc_kv = idesc_bf16(kBK, kD, 0, 1);     // B (Q, dO) MN-major
      constexpr uint32_t idesc_dq = idesc_bf16(kD, kBQ, 1, 1);     // A (K^T), B (dS^T) MN-major
      const uint32_t k_addr = smem_u32(smem + L::kK), v_addr = smem_u32(smem + L::kV);
      bool ok = n_all == 0 || mbar_wait(&bars->kv_full, 0, lim, abort);
      auto issue_grads = [&](int i) -> bool {
        const int st = i % kStages, b = i & 1;
        if (!mbar_wait(&bars->ps_full, i & 1, lim, abort)) return false;
        if (i >= 2 && !mbar_wait(&bars->dq_empty[b], ((i >> 1) - 1) & 1, lim, abort)) return false;
        tc_fence_after();
        const uint32_t p_addr = smem_u32(smem + L::kP);
        const uint32_t ds_addr = smem_u32(smem + L::kDS);
        const uint32_t q_addr = smem_u32(smem + L::kQ + st * 2 * L::kQBox);
        const uint32_t do_addr = smem_u32(smem + L::kDO + st * 2 * L::kQBox);
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk) {     // over queries
          const uint64_t pa = sdesc_sw128(p_addr + kk * 32, 16, 1024);
          const uint64_t da = sdesc_sw128(ds_addr + kk * 32, 16, 1024);
          const uint64_t ob = sdesc_sw128(do_addr + kk * 16 * 128, L::kQBox, 1024);
          const uint64_t qb = sdesc_sw128(q_addr + kk * 16 * 128, L::kQBox, 1024);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          mma_bf16(tmem + kColDV, pa, ob, idesc_kv, acc);
          mma_bf16(tmem + kColDK, da, qb, idesc_kv, acc);
        }
        const uint32_t dsl_addr = smem_u32(smem + L::kDSL);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {     // over keys
          const uint64_t ka = sdesc_sw128(k_addr + kk * 16 * 128, L::kKVBox, 1024);
          const uint64_t sb = sdesc_sw128(ds_addr + kk * 16 * 128, 16, 1024);
          const uint64_t lb = sdesc_sw128(dsl_addr + kk * 16 * 128, 16, 1024);
          mma_bf16(tmem + (b ? kColDQ1 : kColDQ0), ka, sb, idesc_dq, kk > 0 ? 1u : 0u);
          if (kSplit) mma_bf16(tmem + (b ? kColDQ1 : kColDQ0), ka, lb, idesc_dq, 1u);
        }
        mma_commit(&bars->qdo_empty[st]);
        mma_commit(&bars->ps_empty);
        mma_commit(&bars->dq_full[b]);
        return true;
      };
      for (int i = 0; ok && i < n_all; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(&bars->qdo_full[st], (i / kStages) & 1, lim, abort) ||
            (i >= 1 && !mbar_wait(&bars->sdp_empty, (i - 1) & 1, lim, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t q_addr = smem_u32(smem + L::kQ + st * 2 * L::kQBox);
        const uint32_t do_addr = smem_u32(smem + L::kDO + st * 2 * L::kQBox);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {      // over head dim
          const uint32_t ko = (kk / 4) * L::kKVBox + (kk % 4) * 32;
          const uint32_t qo = (kk / 4) * L::kQBox + (kk % 4) * 32;
          mma_bf16(tmem + kColS, sdesc_sw128(k_addr + ko, 16, 1024),
                   sdesc_sw128(q_addr + qo, 16, 1024), idesc_sdp, kk > 0 ? 1u : 0u);
          mma_bf16(tmem + kColDP, sdesc_sw128(v_addr + ko, 16, 1024),
                   sdesc_sw128(do_addr + qo, 16, 1024), idesc_sdp, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->sdp_full);
        if (i >= 1 && !issue_grads(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && n_all > 0 && !issue_grads(n_all - 1)) ok = false;
      if (ok && n_all > 0) mma_commit(&bars->dkv_done);
      if (!ok) {
        record_timeout(a.status, abort, 12);
        mma_commit(&bars->drain);
        int zero = 0;
        mbar_wait(&bars->drain, 0, kDrainLimit, &zero);
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ drain
    // thread = head-dim index (warp & 3) * 32 + lane == TMEM lane of dQ^T.
    // Each tile's dQ^T goes out in four rounds of 16 query columns: the four
    // warps stage them as fp32 [16 rows][128] in shared memory; warp 3 adds
    // each staged block into dQ with a bulk tensor reduce (the reduction runs
    // in L2; no per-thread atomics).
    const int dd = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    constexpr int N = L::kNumStg;
    bool ok = true;
    int k = 0;                                   // round counter
    for (int j = 0; ok && j < n_all; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&bars->dq_full[b], (j >> 1) & 1, lim, abort)) { ok = false; break; }
      tc_fence_after();
      // the whole dQ^T tile (64 query columns) into registers first, so its
      // TMEM buffer is free for the next dQ product before any staging
      uint32_t r[2][32];
      tmem_ld32(tmem + lane_off + (b ? kColDQ1 : kColDQ0), r[0]);
      tmem_ld32(tmem + lane_off + (b ? kColDQ1 : kColDQ0) + 32, r[1]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->dq_empty[b]);
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4, ++k) {
        const int sb = k % N;
        if (k >= N && !mbar_wait(&bars->stg_free[sb], ((k / N) - 1) & 1, lim, abort)) {
          ok = false;
          break;
        }
        float* stg = reinterpret_cast<float*>(smem + L::kStg + sb * L::kStgBytes);
#pragma unroll
        for (int x = 0; x < L::kStgRows; ++x)
          stg[x * kD + dd] = __uint_as_float(r[r4 >> 1][(r4 & 1) * 16 + x]) * a.scale;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->stg_full[sb]);
      }
    }
    if (!ok) record_timeout(a.status, abort, 14);
  } else if (warp == 3) {
    // ------------------------------------------------------------ dQ reduce issue
    // One thread, alone in its warp (a waiting thread never holds up a warp
    // that stages): round k of the drain is staged in buffer k % N.
    if (lane == 0) {
      constexpr int N = L::kNumStg;
      bool ok = true;
      int k = 0;
      int jt = 0, hq = hk * G + (kShared ? blockIdx.x / a.n_items % a.kv_split * Gs : 0);
      for (int j = 0; ok && j < n_all; ++j, jt = jt + 1 == n_qt ? 0 : jt + 1, hq += jt == 0) {
        Seg sgd;
        int q0d, td;
        tile_of(it, jt, sgd, q0d, td);
        const int grow = sgd.row0 + q0d + td * kBQ;   // natural row of the tile's first query
        for (int r4 = 0; r4 < 4; ++r4, ++k) {
          const int sb = k % N;
          if (!mbar_wait(&bars->stg_full[sb], (k / N) & 1, lim, abort)) {
            ok = false;
            break;
          }
          // rows past the run carry exact zeros (P = 0 there); rows past T are
          // clipped by the tensor map
          if (CP_IN_RANGE(grow, 0, a.T, a.status, 305) && CP_IN_RANGE(hq, 0, a.H, a.status, 306)) {
            tma_reduce_add_3d(&a.tm_dq, smem + L::kStg + sb * L::kStgBytes, 0, hq,
                              grow + r4 * L::kStgRows);
          }
          bulk_commit();
          // free this round's buffer as soon as the reduce has read it, so the
          // staging warps can run up to N rounds ahead of this thread
          bulk_wait_read<0>();
          mbar_arrive(&bars->stg_free[sb]);
        }
      }
      bulk_wait_all();                           // every reduce-add finished before exit
      if (!ok) record_timeout(a.status, abort, 15);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P / dS
    // Two warpgroups share every query tile: warpgroup g (warps 4+4g .. 7+4g)
    // computes P^T / dS^T for query columns [32g, 32g + 32) of its key rows.
    const int g = (warp - 4) >> 2;
    const int u = (warp & 3) * 32 + lane;        // key row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    const bool key_ok = u < it.k_len;
    bool ok = true;
    for (int i = 0, jt = 0; ok && i < n_all; ++i, jt = jt + 1 == n_qt ? 0 : jt + 1) {
      Seg sg;
      int q0, t;
      tile_of(it, jt, sg, q0, t);
      const int st = i % kStages;
      if (!mbar_wait(&bars->sdp_full, i & 1, lim, abort) ||
          !mbar_wait(&bars->qdo_full[st], (i / kStages) & 1, lim, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t rs[32], rd[32];
      tmem_ld32(tmem + lane_off + kColS + g * 32, rs);
      tmem_ld32(tmem + lane_off + kColDP + g * 32, rd);
      tmem_ld_wait();
      reg_fence32(rs);
      reg_fence32(rd);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->sdp_empty);
      const int row0 = q0 + t * kBQ + g * 32;     // first query of this half (inside the run)
      const float* ld = reinterpret_cast<const float*>(smem + L::kLd + st * 1024) +
                        ((sg.row0 + q0 + t * kBQ) & 3) + g * 32;
      // key u is visible to query row0 + x iff x < len - row0 and, for a causal
      // run, u <= row0 + x + delta
      const int first_vis = sg.causal ? u - sg.delta - row0 : 0;
      const int end_vis = key_ok ? sg.len - row0 : 0;
      const bool whole = __all_sync(0xffffffffu, first_vis <= 0 && end_vis >= 32);
      uint32_t pk[16], hk[16], lk[16];
      // lse2 / D of the 32 queries: every thread reads the same words, so
      // 16-byte loads (when the tile starts on a 4-row boundary) cut the
      // shared-memory wavefronts four-fold
      auto compute = [&](auto masked, auto vec) {
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          float l[4], dd[4];
          if (decltype(vec)::value) {
            const float4 l4 = *reinterpret_cast<const float4*>(ld + x);
            const float4 d4 = *reinterpret_cast<const float4*>(ld + kLdRows + x);
            l[0] = l4.x; l[1] = l4.y; l[2] = l4.z; l[3] = l4.w;
            dd[0] = d4.x; dd[1] = d4.y; dd[2] = d4.z; dd[3] = d4.w;
          } else {
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              l[y] = ld[x + y];
              dd[y] = ld[kLdRows + x + y];
            }
          }
#pragma unroll
          for (int y = 0; y < 4; y += 2) {
            float p0 = ex2(fmaf(__uint_as_float(rs[x + y]), sl2, -l[y]));
            float p1 = ex2(fmaf(__uint_as_float(rs[x + y + 1]), sl2, -l[y + 1]));
            if (decltype(masked)::value) {
              if (x + y < first_vis || x + y >= end_vis) p0 = 0.f;
              if (x + y + 1 < first_vis || x + y + 1 >= end_vis) p1 = 0.f;
            }
            const float d0 = p0 * (__uint_as_float(rd[x + y]) - dd[y]);
            const float d1 = p1 * (__uint_as_float(rd[x + y + 1]) - dd[y + 1]);
            pk[(x + y) / 2] = pack_bf16x2(p0, p1);
            if (kSplit) {
              const float h0 = __bfloat162float(__float2bfloat16_rn(d0));
              const float h1 = __bfloat162float(__float2bfloat16_rn(d1));
              hk[(x + y) / 2] = pack_bf16x2(h0, h1);
              lk[(x + y) / 2] = pack_bf16x2(d0 - h0, d1 - h1);
            } else {
              hk[(x + y) / 2] = pack_bf16x2(d0, d1);
            }
          }
        }
      };
      using T_ = std::integral_constant<bool, true>;
      using F_ = std::integral_constant<bool, false>;
      const bool aligned = ((sg.row0 + q0 + t * kBQ) & 3) == 0;
      if (aligned) {
        if (whole) compute(F_(), T_());
        else compute(T_(), T_());
      } else {
        if (whole) compute(F_(), F_());
        else compute(T_(), F_());
      }
      if (i >= 1 && !mbar_wait(&bars->ps_empty, (i - 1) & 1, lim, abort)) {
        ok = false;
        break;
      }
      uint8_t* prow = smem + L::kP + u * 128;
      uint8_t* srow = smem + L::kDS + u * 128;
      uint8_t* lrow = smem + L::kDSL + u * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int sw = ((g * 4 + c) ^ (u & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + sw) =
            make_uint4(pk[c * 4], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
        *reinterpret_cast<uint4*>(srow + sw) =
            make_uint4(hk[c * 4], hk[c * 4 + 1], hk[c * 4 + 2], hk[c * 4 + 3]);
        if (kSplit)
          *reinterpret_cast<uint4*>(lrow + sw) =
              make_uint4(lk[c * 4], lk[c * 4 + 1], lk[c * 4 + 2], lk[c * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ps_full);
    }
    // ------------------------------------------------------------ dK / dV epilogue
    if (ok && n_all > 0 && !mbar_wait(&bars->dkv_done, 0, lim, abort)) ok = false;
    // dK / dV rows accumulate over ring steps: the previous step's grid must
    // be complete (a no-op unless launched as a programmatic dependent)
    griddep_wait();
    if (!ok) {
      record_timeout(a.status, abort, 13);
    } else {
      tc_fence_after();
      // warpgroup 0 writes dK (scaled), warpgroup 1 writes dV
      float* dst;
      bool row_ok = key_ok && CP_IN_RANGE(hk, 0, a.Hkv, a.status, 307);
      if (it.dk_mode == DK_TEXT) {
        row_ok = row_ok && CP_IN_RANGE(it.k_row0 + u, 0, a.T, a.status, 308);
        dst = (g == 0 ? a.dk : a.dv) + ((long long)(it.k_row0 + u) * a.Hkv + hk) * kD;
      } else {
        row_ok = row_ok && CP_IN_RANGE(it.slot, 0, a.n_slots, a.status, 309) &&
                 CP_IN_RANGE(it.dk_row0 + u, 0, a.pre_rows, a.status, 310);
        const long long row = (long long)it.slot * a.pre_rows + it.dk_row0 + u;
        dst = (g == 0 ? a.pre_k : a.pre_v) + (row * a.Hkv + hk) * kD;
      }
      const bool first = (it.flags & F_FIRST) != 0;
      const float mul = g == 0 ? a.scale : 1.f;
      const uint32_t col = g == 0 ? kColDK : kColDV;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
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

template <bool kSplit, bool kShared>
cudaError_t launch_split(const TcBwdArgs& a, cudaStream_t st) {
  constexpr int smem = Lay<kSplit>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_kernel<kSplit, kShared>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.n_items * a.Hkv * a.kv_split;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
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
  return cudaLaunchKernelEx(&cfg, tc_bwd_kernel<kSplit, kShared>, a);
}

}  // namespace

cudaError_t launch_tc_bwd(const TcBwdArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  if (a.d != kD) return cudaErrorNotSupported;
  if (a.kv_split < 1 || (a.H / a.Hkv) % a.kv_split != 0) return cudaErrorInvalidValue;
  // The dQ error from one bf16 rounding of dS grows with the softmax scale
  // (dQ = scale * dS K).  Above kPrecisionSplitScale the remainder term is
  // added; every other case runs the 128-query kernel (tc_bwd_q128.cu).
  if (!(a.scale > kPrecisionSplitScale)) return cudaErrorNotSupported;
  return a.kv_split > 1 ? launch_split<true, true>(a, st) : launch_split<true, false>(a, st);
}

}  // namespace cpattn
