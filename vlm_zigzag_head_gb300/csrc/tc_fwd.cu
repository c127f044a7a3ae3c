// Ring-step attention forward on 5th-generation tensor cores (sm_103a).
//
// One CTA computes one work item of a ring step for one head: a tile of 128
// query rows against the key runs the step gives it (page
// "context-parallel-multimodal": §1.1 zigzag chunks, §1 ring order, §4.1
// replicated prefix in step 0), with an online softmax over the KV tiles and
// a fused log-sum-exp merge into the fp32 running result (or the final write
// in natural order).
//
// Warp roles (384 threads; TMEM lane quarter of warp w is w % 4):
//   warp 0       TMA producer of Q and K tiles
//   warp 1       TMEM allocation; lane 0 issues every tcgen05.mma
//   warp 2       TMA producer of V tiles
//   warp 3       idle
//   warps 4..7   softmax of key columns 0..63 of every S tile, then the
//                epilogue of O columns [0, D/2); thread = query row = TMEM lane
//   warps 8..11  the same for key columns 64..127 and O columns [D/2, D)
// The two warps that share a query row exchange their partial row maxima
// (and, at the end, their partial row sums) through shared memory; a per-pair
// mbarrier (bounded waits, like every other wait here) orders the exchange.
//
// TMEM (512 columns): S ping-pong buffers at columns [0,128) and [128,256),
// the O accumulator at [256, 256 + D), Q as bf16 pairs at [384, 384 + D/2).
// P (bf16) overwrites the S buffer it was computed from: the warp of key
// half g writes its 64 probabilities at buffer columns [64g, 64g + 32).  Both
// products read their A operand (Q, P) from TMEM and only B (K, V) from
// shared memory.  Shared memory: Q (128 x D), two K and two V stages
// (128 x D each), in the 128-byte swizzled layout TMA writes.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc.h"

namespace cpattn {

namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kBM = kFwdTileQ;   // 128 query rows
constexpr int kBN = kFwdTileK;   // 128 keys per KV tile
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColQ = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max may lag by 2^8
constexpr long long kDrainLimit = 1LL << 24;

template <int D>
struct Smem {
  static constexpr int kTile = kBM * D * 2;        // bytes of a 128 x D bf16 tile
  static constexpr int kBox = 128 * 128;           // one 128-row x 128-byte TMA box
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;
  static constexpr int kXch = kP;                       // [parity][half][128] float exchange
  static constexpr int kBars = kXch + 4 * kBM * 4;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2];
  uint64_t q_tmem;    // Q copied into TMEM by the softmax warps
  uint64_t p_full, o_done;
  uint64_t drain;
  uint64_t pair[4];   // the two softmax warps of each TMEM lane quarter
  uint32_t tmem_base;
  int abort;
};

// Tiles of one key run visible to a query tile of q_len rows.
__device__ __forceinline__ int run_tiles(const Seg& s, int q_len) {
  int vis = s.len;
  if (s.causal) {
    vis = q_len + s.delta;
    vis = vis < 0 ? 0 : (vis < s.len ? vis : s.len);
  }
  return (vis + kBN - 1) / kBN;
}

__device__ __forceinline__ void record_timeout(int32_t* status, volatile int* abort, int site) {
  if (atomicCAS(&status[0], 0, 1) == 0) status[1] = site;
  *abort = 1;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ TcFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps shared-space (not generic) loads and stores
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  using L = Smem<D>;
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_idx = blockIdx.x % a.n_items;
  const int h = blockIdx.x / a.n_items;
  const FwdItem& it = a.items[item_idx];
  volatile int* abort = &bars->abort;
  const long long lim = a.wait_limit;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&bars->s_full[b], 1);
    mbar_init(&bars->q_tmem, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&bars->pair[q], 2);
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

  const int q_len = it.q_len;
  const int nseg = it.nseg;
  int n_tiles = 0;
  for (int s = 0; s < nseg; ++s) n_tiles += run_tiles(it.seg[s], q_len);

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const bool is_k = warp == 0;
      int issued = 0;  // tiles issued by this producer
      bool q_issued = false;
      if (is_k && n_tiles > 0) {
        const CUtensorMap* qm = it.q_src == SRC_TEXT ? &a.tm_q_text : &a.tm_q_nat;
        mbar_expect_tx(&bars->q_full, L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(qm, &bars->q_full, smem + L::kQ + b * L::kBox, b * 64, h, it.q_row0);
        q_issued = true;
      }
      int j = 0;
      for (int s = 0; s < nseg && !*abort; ++s) {
        const Seg sg = it.seg[s];
        const CUtensorMap* m = is_k ? (sg.src == SRC_TEXT ? &a.tm_k_text : &a.tm_k_nat)
                                    : (sg.src == SRC_TEXT ? &a.tm_v_text : &a.tm_v_nat);
        const int nt = run_tiles(sg, q_len);
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
            tma_load_3d(m, full, dst + b * L::kBox, b * 64, h, sg.row0 + t * kBN);
          issued = j + 1;
        }
        if (*abort) break;
      }
      // every load this producer issued must land before the CTA exits
      // (normally the MMA issuer already waited for them: these return at once)
      {
        int zero = 0;
        if (q_issued) mbar_wait(&bars->q_full, 0, kDrainLimit, &zero);
        for (int x = issued - kStages; x < issued; ++x) {
          if (x < 0) continue;
          const int st = x % kStages;
          uint64_t* full = is_k ? &bars->k_full[st] : &bars->v_full[st];
          mbar_wait(full, (x / kStages) & 1, kDrainLimit, &zero);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, D, 0, 1);
      bool ok = n_tiles == 0 || mbar_wait(&bars->q_tmem, 0, lim, abort);
      if (!ok) record_timeout(a.status, abort, 3);
      auto issue_pv = [&](int i) -> bool {
        const int st = i % kStages;
        if (!mbar_wait(&bars->p_full, i & 1, lim, abort)) return false;
        if (!mbar_wait(&bars->v_full[st], (i / kStages) & 1, lim, abort)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + L::kV + st * L::kTile);
        const uint32_t p_tmem = tmem + ((i & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {   // keys 16kk..: half kk/4, column (kk%4)*8
          const uint64_t bd = sdesc_sw128(v_addr + kk * 16 * 128, L::kBox, 1024);
          mma_bf16_ts(tmem + kColO, p_tmem + (kk / 4) * 64 + (kk % 4) * 8, bd, idesc_pv,
                      (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->v_empty[st]);
        mma_commit(&bars->o_done);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % kStages, sb = j & 1;
        // the S buffer of tile j last held P_{j-2}, read by PV_{j-2}, issued
        // (and so executed) before this product
        if (!mbar_wait(&bars->k_full[st], (j / kStages) & 1, lim, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + L::kK + st * L::kTile);
        const uint32_t s_tmem = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {     // head dims 16kk..: Q columns 8kk..
          const uint32_t off = (kk / 4) * L::kBox + (kk % 4) * 32;
          mma_bf16_ts(s_tmem, tmem + kColQ + kk * 8, sdesc_sw128(k_addr + off, 16, 1024),
                      idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->k_empty[st]);
        mma_commit(&bars->s_full[sb]);
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && n_tiles > 0 && !issue_pv(n_tiles - 1)) ok = false;
      if (!ok) {
        record_timeout(a.status, abort, 4);
        // drain: nothing issued by this thread may still be running at exit
        mma_commit(&bars->drain);
        int zero = 0;
        mbar_wait(&bars->drain, 0, kDrainLimit, &zero);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int g = (warp - 4) >> 2;             // key-column half of S / O-column half
    const int t = (warp & 3) * 32 + lane;      // query row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    uint64_t* pair = &bars->pair[warp & 3];
    float* xch = reinterpret_cast<float*>(smem + L::kXch);  // [parity][half][128]
    // exchange a per-row value with the partner warp; phase k of the pair barrier
    auto exchange = [&](float v, int k, float* partner) -> bool {
      xch[((k & 1) * 2 + g) * kBM + t] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(pair);
      if (!mbar_wait(pair, k & 1, lim, abort)) return false;
      *partner = xch[((k & 1) * 2 + (1 - g)) * kBM + t];
      return true;
    };
    const float sl2 = a.scale_log2;
    float m = -INFINITY;   // running max of scaled scores (log2 units), may lag
    float l = 0.f;         // partial row sum over this thread's columns
    bool ok = true;
    // Q row t into TMEM (bf16 pairs): warp half g copies head dims [64g, 64g + 64)
    if (n_tiles > 0) {
      if (!mbar_wait(&bars->q_full, 0, lim, abort)) ok = false;
      if (ok && g * 64 < D) {
        uint32_t r[32];
        const uint8_t* qrow = smem + L::kQ + g * L::kBox + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((c ^ (t & 7)) << 4));
          r[c * 4 + 0] = v.x;
          r[c * 4 + 1] = v.y;
          r[c * 4 + 2] = v.z;
          r[c * 4 + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kColQ + g * 32, r);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_tmem);
    }
    int j = 0;
    for (int s = 0; ok && s < nseg; ++s) {
      const Seg sg = it.seg[s];
      const int nt = run_tiles(sg, q_len);
      for (int tt = 0; tt < nt; ++tt, ++j) {
        const int sb = j & 1;
        if (!mbar_wait(&bars->s_full[sb], (j >> 1) & 1, lim, abort)) { ok = false; break; }
        tc_fence_after();
        constexpr int kH = kBN / 2;              // 64 columns per thread
        float x[kH];
        {
          uint32_t r[kH];
          const uint32_t s_col = tmem + lane_off + (sb ? kColS1 : kColS0) + g * kH;
#pragma unroll
          for (int c = 0; c < kH / 32; ++c)
            tmem_ld32(s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kH / 32; ++c)
            reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
#pragma unroll
          for (int c = 0; c < kH; ++c) x[c] = __uint_as_float(r[c]) * sl2;
        }
        // mask: key u = u0 + c visible iff u < len and (!causal or u <= t + delta)
        const int u0 = tt * kBN + g * kH;
        const bool full = (u0 + kH <= sg.len) && (!sg.causal || u0 + kH - 1 <= sg.delta);
        if (!full) {
          const int lim_u = sg.causal ? min(sg.len, t + sg.delta + 1) : sg.len;
#pragma unroll
          for (int c = 0; c < kH; ++c)
            if (u0 + c >= lim_u) x[c] = -INFINITY;
        }
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = x[i];
#pragma unroll
        for (int c = 8; c < kH; ++c) mp[c & 7] = fmaxf(mp[c & 7], x[c]);
        float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                         fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        // combine with the partner half of the row (same value in both threads)
        float mo;
        if (!exchange(mt, j, &mo)) { ok = false; break; }
        mt = fmaxf(mt, mo);
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold || (m == -INFINITY && m_new != -INFINITY);
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m - m_new) : 1.f;  // m = -inf -> 0
          if (need) {
            l *= alpha;
            m = m_new;
          }
          if (j > 0) {  // O holds PV of earlier tiles: wait for the last, rescale our half
            if (!mbar_wait(&bars->o_done, (j - 1) & 1, lim, abort)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
              uint32_t r[32];
              const uint32_t col = tmem + lane_off + kColO + g * (D / 2) + c * 32;
              tmem_ld32(col, r);
              tmem_ld_wait();
              reg_fence32(r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(col, r);
            }
            tmem_st_wait();
          }
        }
        const float mu = m == -INFINITY ? 0.f : m;
        float sp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sp[i] = 0.f;
#pragma unroll
        for (int c = 0; c < kH; ++c) {
          x[c] = ex2(x[c] - mu);
          sp[c & 7] += x[c];
        }
        l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        // P (bf16 pairs) over this thread's own S columns: buffer columns
        // [64g, 64g + 32); PV_j reads it from there
        {
          uint32_t pk[kH / 2];
#pragma unroll
          for (int c = 0; c < kH / 2; ++c) pk[c] = pack_bf16x2(x[2 * c], x[2 * c + 1]);
          tmem_st32(tmem + lane_off + (sb ? kColS1 : kColS0) + g * 64, pk);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0 && !mbar_wait(&bars->o_done, (n_tiles - 1) & 1, lim, abort)) ok = false;
    // the row's two partial sums
    float lo_part = 0.f;
    if (ok && !exchange(l, n_tiles, &lo_part)) ok = false;
    l += lo_part;
    if (!ok) {
      record_timeout(a.status, abort, 5);
    } else {
      tc_fence_after();
      const bool valid = t < q_len;
      float lse_s = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int flags = it.flags;
      const long long rrow =
          it.run_row0 >= 0 ? (long long)h * a.run_rows + it.run_row0 + t : 0;
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
      const int c0 = g * (D / 2);               // this thread's O columns
      const float* orun = a.o_run + rrow * D + c0;
      float* orun_w = a.o_run + rrow * D + c0;
      const long long out_off = ((long long)(it.out_row0 + t) * a.H + h) * D + c0;
      __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(a.out) + out_off;
      __nv_bfloat16* lop =
          a.out_lo ? reinterpret_cast<__nv_bfloat16*>(a.out_lo) + out_off : nullptr;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kColO + c0 + c * 32, r);
        tmem_ld_wait();
        reg_fence32(r);
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
      if (valid && g == 0) {
        if (flags & F_FINAL) a.lse[(long long)h * a.T + it.out_row0 + t] = lse_s;
        else a.lse_run[rrow] = lse_s;
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

template <int D>
cudaError_t launch_d(const TcFwdArgs& a, cudaStream_t st) {
  const int smem = Smem<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.n_items * a.H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  tc_fwd_kernel<D><<<(unsigned)blocks, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd(const TcFwdArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  return a.d == 64 ? launch_d<64>(a, st) : launch_d<128>(a, st);
}

}  // namespace cpattn
