// CUDA-core attention for fp32 inputs (FFMA, accurate expf/logf), the parity
// path of the fp32 interface (bf16 inputs always run on the tensor cores): one
// work item of the ring-step plan per block.  It walks the same work lists as the
// tensor-core kernels: a query tile against runs of keys (forward, dQ), or a
// key tile against runs of queries (dK, dV).
#include <cuda_bf16.h>

#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kSimtQ = 128;   // query rows per block (one per thread)
constexpr int kSimtKT = 32;   // keys staged per round
constexpr int kSimtQT = 32;   // queries staged per round (dK/dV pass)
constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_f(T* p, float x);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ int seg_visible_keys(const Seg& s, int q_len) {
  if (!s.causal) return s.len;
  const int v = q_len + s.delta;
  return v < 0 ? 0 : (v < s.len ? v : s.len);
}

// ---------------------------------------------------------------------------
// forward: query tile x key runs, online softmax, then the log-sum-exp merge
// into the running result (or the final natural-order write)
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kSimtQ) simt_fwd_kernel(SimtFwdArgs a) {
  extern __shared__ float smem[];
  float* Qs = smem;                        // [kSimtQ][D + 1]
  float* Ks = Qs + kSimtQ * (D + 1);       // [kSimtKT][D]
  float* Vs = Ks + kSimtKT * D;            // [kSimtKT][D]
  __shared__ FwdItem it;
  const int h = blockIdx.y;
  const int t = threadIdx.x;
  if (t == 0) it = a.items[blockIdx.x];
  __syncthreads();
  const int H = a.H;
  const int Hkv = a.Hkv, hk = h / (H / Hkv);   // the KV head this query head reads
  const T* qsrc = static_cast<const T*>(it.q_src == SRC_TEXT ? a.q_text : a.q_nat);
  for (int x = t; x < kSimtQ * D; x += kSimtQ) {
    const int row = x / D, e = x - row * D;
    Qs[row * (D + 1) + e] =
        row < it.q_len ? ld_f(qsrc + ((long long)(it.q_row0 + row) * H + h) * D + e) : 0.f;
  }
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;
  const bool valid = t < it.q_len;
  for (int sg = 0; sg < it.nseg; ++sg) {
    const Seg s = it.seg[sg];
    const T* ksrc = static_cast<const T*>(s.src == SRC_TEXT ? a.k_text : a.k_nat);
    const T* vsrc = static_cast<const T*>(s.src == SRC_TEXT ? a.v_text : a.v_nat);
    const int nkeys = seg_visible_keys(s, it.q_len);
    for (int u0 = 0; u0 < nkeys; u0 += kSimtKT) {
      __syncthreads();
      for (int x = t; x < kSimtKT * D; x += kSimtQ) {
        const int u = x / D, e = x - u * D;
        const bool in = u0 + u < nkeys;
        const long long g = ((long long)(s.row0 + u0 + u) * Hkv + hk) * D + e;
        Ks[x] = in ? ld_f(ksrc + g) : 0.f;
        Vs[x] = in ? ld_f(vsrc + g) : 0.f;
      }
      __syncthreads();
      if (!valid) continue;
      float sc[kSimtKT];
      float tmax = -INFINITY;
#pragma unroll 4
      for (int u = 0; u < kSimtKT; ++u) {
        const int uu = u0 + u;
        const bool vis = uu < nkeys && (!s.causal || uu <= t + s.delta);
        float dot = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) dot += Qs[t * (D + 1) + e] * Ks[u * D + e];
        sc[u] = vis ? dot * a.scale : -INFINITY;
        tmax = fmaxf(tmax, sc[u]);
      }
      if (tmax == -INFINITY) continue;
      const float mn = fmaxf(m, tmax);
      const float corr = expf(m - mn);  // m = -inf -> 0
      l *= corr;
#pragma unroll
      for (int e = 0; e < D; ++e) acc[e] *= corr;
      m = mn;
#pragma unroll 2
      for (int u = 0; u < kSimtKT; ++u) {
        const float p = expf(sc[u] - m);
        l += p;
#pragma unroll
        for (int e = 0; e < D; ++e) acc[e] += p * Vs[u * D + e];
      }
    }
  }
  if (!valid) return;
  // partial of this ring step
  float lse_s = l > 0.f ? m + logf(l) : -INFINITY;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] *= inv;
  const long long rrow = it.run_row0 >= 0 ? (long long)h * a.run_rows + it.run_row0 + t : 0;
  if (!(it.flags & F_FIRST)) {  // log-sum-exp merge with the running result
    const float lr = a.lse_run[rrow];
    const float mm = fmaxf(lr, lse_s);
    if (mm != -INFINITY) {
      const float wa = expf(lr - mm), wb = expf(lse_s - mm), tot = wa + wb;
      const float ca = wa / tot, cb = wb / tot;
      const float* orun = a.o_run + rrow * D;
#pragma unroll
      for (int e = 0; e < D; ++e) acc[e] = ca * orun[e] + cb * acc[e];
      lse_s = mm + logf(tot);
    }
  }
  if (it.flags & F_FINAL) {
    T* out = static_cast<T*>(a.out) + ((long long)(it.out_row0 + t) * H + h) * D;
#pragma unroll
    for (int e = 0; e < D; ++e) st_f(out + e, acc[e]);
    a.lse[(long long)h * a.T + it.out_row0 + t] = lse_s;
  } else {
    float* orun = a.o_run + rrow * D;
#pragma unroll
    for (int e = 0; e < D; ++e) orun[e] = acc[e];
    a.lse_run[rrow] = lse_s;
  }
}

// ---------------------------------------------------------------------------
// backward dQ: query tile x key runs with the final lse (natural order)
// dQ_t = scale sum_u P_tu (dO_t . v_u - D_t) k_u
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kSimtQ) simt_bwd_dq_kernel(SimtBwdArgs a, int first_item) {
  extern __shared__ float smem[];
  float* Qs = smem;                        // [kSimtQ][D + 1]
  float* dOs = Qs + kSimtQ * (D + 1);      // [kSimtQ][D + 1]
  float* Ks = dOs + kSimtQ * (D + 1);      // [kSimtKT][D]
  float* Vs = Ks + kSimtKT * D;            // [kSimtKT][D]
  __shared__ FwdItem it;
  const int h = blockIdx.y;
  const int t = threadIdx.x;
  if (t == 0) it = a.q_items[first_item + blockIdx.x];
  __syncthreads();
  const int H = a.H;
  const int Hkv = a.Hkv, hk = h / (H / Hkv);   // the KV head this query head reads
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  for (int x = t; x < kSimtQ * D; x += kSimtQ) {
    const int row = x / D, e = x - row * D;
    const bool in = row < it.q_len;
    const long long g = ((long long)(it.q_row0 + row) * H + h) * D + e;
    Qs[row * (D + 1) + e] = in ? ld_f(q + g) : 0.f;
    dOs[row * (D + 1) + e] = in ? ld_f(dout + g) : 0.f;
  }
  const bool valid = t < it.q_len;
  const long long qrow = it.q_row0 + t;
  const float lse2 = valid ? a.lse2[(long long)h * a.pitch + qrow] : 0.f;
  const float Dt = valid ? a.D[(long long)h * a.pitch + qrow] : 0.f;
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  for (int sg = 0; sg < it.nseg; ++sg) {
    const Seg s = it.seg[sg];
    const int nkeys = seg_visible_keys(s, it.q_len);
    for (int u0 = 0; u0 < nkeys; u0 += kSimtKT) {
      __syncthreads();
      for (int x = t; x < kSimtKT * D; x += kSimtQ) {
        const int u = x / D, e = x - u * D;
        const bool in = u0 + u < nkeys;
        const long long g = ((long long)(s.row0 + u0 + u) * Hkv + hk) * D + e;
        Ks[x] = in ? ld_f(k + g) : 0.f;
        Vs[x] = in ? ld_f(v + g) : 0.f;
      }
      __syncthreads();
      if (!valid) continue;
      for (int u = 0; u < kSimtKT; ++u) {
        const int uu = u0 + u;
        if (!(uu < nkeys && (!s.causal || uu <= t + s.delta))) continue;
        float dk = 0.f, dv = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) {
          dk += Qs[t * (D + 1) + e] * Ks[u * D + e];
          dv += dOs[t * (D + 1) + e] * Vs[u * D + e];
        }
        const float p = exp2f(dk * a.scale * kLog2e - lse2);
        const float ds = p * (dv - Dt) * a.scale;
#pragma unroll
        for (int e = 0; e < D; ++e) acc[e] += ds * Ks[u * D + e];
      }
    }
  }
  if (!valid) return;
  float* dst = a.dq + (qrow * H + h) * D;
  if (it.flags & F_FIRST) {
#pragma unroll
    for (int e = 0; e < D; ++e) dst[e] = acc[e];
  } else {
#pragma unroll
    for (int e = 0; e < D; ++e) dst[e] += acc[e];
  }
}

// ---------------------------------------------------------------------------
// backward dK/dV: key tile x query runs.  Two threads per key (each owns half
// of d); partial dot products are combined with one shuffle.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(2 * kBwdTileK) simt_bwd_dkdv_kernel(SimtBwdArgs a,
                                                                      int first_item) {
  constexpr int HD = D / 2;
  extern __shared__ float smem[];
  float* Ks = smem;                          // [kBwdTileK][D + 1]
  float* Vs = Ks + kBwdTileK * (D + 1);      // [kBwdTileK][D + 1]
  float* Qs = Vs + kBwdTileK * (D + 1);      // [kSimtQT][D]
  float* dOs = Qs + kSimtQT * D;             // [kSimtQT][D]
  float* Ls = dOs + kSimtQT * D;             // [kSimtQT]
  float* Dsm = Ls + kSimtQT;                 // [kSimtQT]
  __shared__ BwdItem it;
  const int hk = blockIdx.y;                 // KV head; its query heads are hk*G .. hk*G+G-1
  const int tid = threadIdx.x;
  const int u = tid >> 1, half = tid & 1;
  if (tid == 0) it = a.k_items[first_item + blockIdx.x];
  __syncthreads();
  const int H = a.H, Hkv = a.Hkv, G = H / Hkv;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  for (int x = tid; x < kBwdTileK * D; x += 2 * kBwdTileK) {
    const int row = x / D, e = x - row * D;
    const bool in = row < it.k_len;
    const long long g = ((long long)(it.k_row0 + row) * Hkv + hk) * D + e;
    Ks[row * (D + 1) + e] = in ? ld_f(k + g) : 0.f;
    Vs[row * (D + 1) + e] = in ? ld_f(v + g) : 0.f;
  }
  float dk[HD], dv[HD];
#pragma unroll
  for (int e = 0; e < HD; ++e) dk[e] = dv[e] = 0.f;
  const bool valid = u < it.k_len;
  for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi;
    for (int sg = 0; sg < it.nseg; ++sg) {
      const Seg s = it.seg[sg];
      const int t_begin = s.causal ? (s.delta < 0 ? -s.delta : 0) : 0;
      for (int t0 = t_begin; t0 < s.len; t0 += kSimtQT) {
        __syncthreads();
        for (int x = tid; x < kSimtQT * D; x += 2 * kBwdTileK) {
          const int row = x / D, e = x - row * D;
          const bool in = t0 + row < s.len;
          const long long g = ((long long)(s.row0 + t0 + row) * H + h) * D + e;
          Qs[x] = in ? ld_f(q + g) : 0.f;
          dOs[x] = in ? ld_f(dout + g) : 0.f;
        }
        for (int x = tid; x < kSimtQT; x += 2 * kBwdTileK) {
          const bool in = t0 + x < s.len;
          const long long g = (long long)h * a.pitch + s.row0 + t0 + x;
          Ls[x] = in ? a.lse2[g] : 0.f;
          Dsm[x] = in ? a.D[g] : 0.f;
        }
        __syncthreads();
        for (int tq = 0; tq < kSimtQT; ++tq) {
          const int tt = t0 + tq;
          float pk = 0.f, pv = 0.f;
#pragma unroll 8
          for (int e = 0; e < HD; ++e) {
            pk += Qs[tq * D + half * HD + e] * Ks[u * (D + 1) + half * HD + e];
            pv += dOs[tq * D + half * HD + e] * Vs[u * (D + 1) + half * HD + e];
          }
          pk += __shfl_xor_sync(0xffffffffu, pk, 1);
          pv += __shfl_xor_sync(0xffffffffu, pv, 1);
          const bool vis = valid && tt < s.len && (!s.causal || u <= tt + s.delta);
          if (!vis) continue;
          const float p = exp2f(pk * a.scale * kLog2e - Ls[tq]);
          const float ds = p * (pv - Dsm[tq]) * a.scale;
#pragma unroll
          for (int e = 0; e < HD; ++e) {
            dv[e] += p * dOs[tq * D + half * HD + e];
            dk[e] += ds * Qs[tq * D + half * HD + e];
          }
        }
      }
    }
  }
  if (!valid) return;
  float *pk, *pv;
  if (it.dk_mode == DK_TEXT) {
    pk = a.dk + ((long long)(it.k_row0 + u) * Hkv + hk) * D + half * HD;
    pv = a.dv + ((long long)(it.k_row0 + u) * Hkv + hk) * D + half * HD;
  } else {
    const long long row = (long long)it.slot * a.pre_rows + it.dk_row0 + u;
    pk = a.pre_k + (row * Hkv + hk) * D + half * HD;
    pv = a.pre_v + (row * Hkv + hk) * D + half * HD;
  }
  if (it.flags & F_FIRST) {
#pragma unroll
    for (int e = 0; e < HD; ++e) { pk[e] = dk[e]; pv[e] = dv[e]; }
  } else {
#pragma unroll
    for (int e = 0; e < HD; ++e) { pk[e] += dk[e]; pv[e] += dv[e]; }
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t fwd_t(const SimtFwdArgs& a, cudaStream_t st) {
  const size_t sm = sizeof(float) * (kSimtQ * (D + 1) + 2 * kSimtKT * D);
  cudaError_t e = set_smem(simt_fwd_kernel<T, D>, sm);
  if (e != cudaSuccess) return e;
  simt_fwd_kernel<T, D><<<dim3(a.n_items, a.H), kSimtQ, sm, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dq_t(const SimtBwdArgs& a, cudaStream_t st) {
  const size_t sm = sizeof(float) * (2 * kSimtQ * (D + 1) + 2 * kSimtKT * D);
  cudaError_t e = set_smem(simt_bwd_dq_kernel<T, D>, sm);
  if (e != cudaSuccess) return e;
  simt_bwd_dq_kernel<T, D><<<dim3(a.n_q_items, a.H), kSimtQ, sm, st>>>(a, 0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dkdv_t(const SimtBwdArgs& a, cudaStream_t st) {
  const size_t sm =
      sizeof(float) * (2 * kBwdTileK * (D + 1) + 2 * kSimtQT * D + 2 * kSimtQT);
  cudaError_t e = set_smem(simt_bwd_dkdv_kernel<T, D>, sm);
  if (e != cudaSuccess) return e;
  simt_bwd_dkdv_kernel<T, D><<<dim3(a.n_k_items, a.Hkv), 2 * kBwdTileK, sm, st>>>(a, 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fwd(const SimtFwdArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  return a.d == 64 ? fwd_t<float, 64>(a, st) : fwd_t<float, 128>(a, st);
}

cudaError_t launch_simt_bwd_dq(const SimtBwdArgs& a, cudaStream_t st) {
  if (a.n_q_items == 0) return cudaSuccess;
  return a.d == 64 ? dq_t<float, 64>(a, st) : dq_t<float, 128>(a, st);
}

cudaError_t launch_simt_bwd_dkdv(const SimtBwdArgs& a, cudaStream_t st) {
  if (a.n_k_items == 0) return cudaSuccess;
  return a.d == 64 ? dkdv_t<float, 64>(a, st) : dkdv_t<float, 128>(a, st);
}

}  // namespace cpattn
