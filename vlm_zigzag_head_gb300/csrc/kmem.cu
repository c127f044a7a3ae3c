// HBM-bound kernels of the path: zigzag gather/scatter and index tables,
// standalone log-sum-exp merge, backward preprocess, prefix-gradient sum, and
// the power-of-two-scaled f16 operand copies.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

struct RowPtrs {
  const uint4* s0; const uint4* s1; const uint4* s2; const uint4* s3;
  uint4* d0; uint4* d1; uint4* d2; uint4* d3;
};

// One warp moves one row of one tensor; 16-byte vectors, coalesced per row.
// gather: dst[k] = src[idx[k]];  scatter: dst[idx[k]] = src[k].
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(RowPtrs p, int n_tensors,
                                                               int vec_per_row,
                                                               const int32_t* __restrict__ idx,
                                                               int n_rows, int scatter) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kThreads / 32);
  const long long total = (long long)n_rows * n_tensors;
  for (long long w = (long long)blockIdx.x * (kThreads / 32) + threadIdx.x / 32; w < total;
       w += warps) {
    const int tsel = (int)(w % n_tensors);
    const long long k = w / n_tensors;
    const long long ik = idx[k];
    const long long srow = scatter ? k : ik;
    const long long drow = scatter ? ik : k;
    const uint4* s = tsel == 0 ? p.s0 : tsel == 1 ? p.s1 : tsel == 2 ? p.s2 : p.s3;
    uint4* d = tsel == 0 ? p.d0 : tsel == 1 ? p.d1 : tsel == 2 ? p.d2 : p.d3;
    s += srow * vec_per_row;
    d += drow * vec_per_row;
    int e = lane;
    for (; e + 96 < vec_per_row; e += 128) {
      uint4 a = ld_stream(s + e), b = ld_stream(s + e + 32), c = ld_stream(s + e + 64),
            f = ld_stream(s + e + 96);
      d[e] = a;
      d[e + 32] = b;
      d[e + 64] = c;
      d[e + 96] = f;
    }
    for (; e < vec_per_row; e += 32) d[e] = ld_stream(s + e);
  }
}

// Thread per permuted text row of one batch of samples: rank r, then the
// sample by binary search over the batch's rank-local offsets, then chunk r
// or 2P-1-r of that sample (page §1.1 head-tail pairing, §5.3 per sample).
// The batch's sample table travels in the kernel parameters.
__global__ void zigzag_index_kernel(const __grid_constant__ ZigzagBatch b, int32_t* fwd_idx,
                                    int32_t* inv_idx) {
  const long long n = (long long)b.span * b.P;
  for (long long m = (long long)blockIdx.x * blockDim.x + threadIdx.x; m < n;
       m += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(m / b.span);
    const long long loc = b.loc0 + (m - (long long)r * b.span);   // rank-local row
    int lo = 0, hi = b.n - 1;
    while (lo < hi) {  // last sample of the batch whose range [off, off + 2c) starts at or before loc
      const int mid = (lo + hi + 1) >> 1;
      if (b.smp[mid][2] <= loc) lo = mid; else hi = mid - 1;
    }
    while (lo > 0 && b.smp[lo][1] == 0) --lo;  // text-less samples share the next one's offset
    const long long t0 = b.smp[lo][0], c = b.smp[lo][1], off = b.smp[lo][2], ord0 = b.smp[lo][3];
    const long long within = loc - off;
    const int slot = (int)(within / c);
    const long long t = within - slot * c;
    const long long ch = slot == 0 ? r : 2LL * b.P - 1 - r;
    const long long k = (long long)r * b.R + loc;
    if (fwd_idx) fwd_idx[k] = (int32_t)(t0 + ch * c + t);
    if (inv_idx) inv_idx[ord0 + ch * c + t] = (int32_t)k;
  }
}

// One warp per (row, head): fold the parts in index order,
// (o, l) (+) (o_p, l_p) with -inf parts contributing nothing.
__global__ void __launch_bounds__(kThreads) lse_merge_kernel(int n_parts,
                                                             const float* __restrict__ po,
                                                             const float* __restrict__ pl,
                                                             int rows, int H, int d, void* out,
                                                             int out_bf16, float* lse) {
  const int lane = threadIdx.x & 31;
  const long long pairs = (long long)rows * H;
  const long long stride_part_o = (long long)rows * H * d;
  const long long stride_part_l = (long long)rows * H;
  for (long long w = (long long)blockIdx.x * (kThreads / 32) + threadIdx.x / 32; w < pairs;
       w += (long long)gridDim.x * (kThreads / 32)) {
    const int h = (int)(w / rows);
    const long long row = w - (long long)h * rows;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float l_run = -INFINITY;
    for (int p = 0; p < n_parts; ++p) {
      const float lp = pl[p * stride_part_l + (long long)h * rows + row];
      const float m = fmaxf(l_run, lp);
      if (m == -INFINITY) continue;
      const float wa = expf(l_run - m), wb = expf(lp - m);
      const float tot = wa + wb;
      const float ca = wa / tot, cb = wb / tot;
      const float* src = po + p * stride_part_o + (row * H + h) * (long long)d;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = lane + 32 * i;
        if (e < d) acc[i] = ca * acc[i] + cb * src[e];
      }
      l_run = m + logf(tot);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane + 32 * i;
      if (e >= d) continue;
      const long long o = (row * H + h) * (long long)d + e;
      if (out_bf16) reinterpret_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(acc[i]);
      else reinterpret_cast<float*>(out)[o] = acc[i];
    }
    if (lane == 0) lse[(long long)h * rows + row] = l_run;
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// d a multiple of 4: one warp per (row, head), 4 consecutive elements per
// lane (16-byte loads).  The merged lse comes first (max, then the sum of
// exp(lse_p - max), both over the parts in lanes), then every part's row is
// read once with its weight exp(lse_p - lse): the parts' loads do not wait on
// one another.
__global__ void __launch_bounds__(kThreads) lse_merge_v4_kernel(int n_parts,
                                                                const float* __restrict__ po,
                                                                const float* __restrict__ pl,
                                                                int rows, int H, int d, void* out,
                                                                int out_bf16, float* lse) {
  const int lane = threadIdx.x & 31;
  const long long pairs = (long long)rows * H;
  const long long stride_o = (long long)rows * H * d;
  const long long stride_l = (long long)rows * H;
  const bool mine = lane * 4 < d;
  for (long long w = (long long)blockIdx.x * (kThreads / 32) + threadIdx.x / 32; w < pairs;
       w += (long long)gridDim.x * (kThreads / 32)) {
    const int h = (int)(w / rows);
    const long long row = w - (long long)h * rows;
    const float* lp = pl + (long long)h * rows + row;
    float m = -INFINITY;
    for (int p = lane; p < n_parts; p += 32) m = fmaxf(m, lp[p * stride_l]);
    m = warp_max(m);
    const long long o = (row * H + h) * (long long)d + lane * 4;
    if (m == -INFINITY) {   // no part saw a key
      if (mine) {
        if (out_bf16) *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o) =
            make_uint2(0u, 0u);
        else *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) =
            make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (lane == 0) lse[(long long)h * rows + row] = -INFINITY;
      continue;
    }
    float sum = 0.f;
    for (int p = lane; p < n_parts; p += 32) sum += expf(lp[p * stride_l] - m);
    const float l_tot = m + logf(warp_sum(sum));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* src = po + (row * H + h) * (long long)d + lane * 4;
#pragma unroll 4
    for (int p = 0; p < n_parts; ++p) {
      const float wgt = expf(lp[p * stride_l] - l_tot);   // 0 for a part with lse = -inf
      if (mine) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src + p * stride_o));
        acc.x = fmaf(wgt, x.x, acc.x);
        acc.y = fmaf(wgt, x.y, acc.y);
        acc.z = fmaf(wgt, x.z, acc.z);
        acc.w = fmaf(wgt, x.w, acc.w);
      }
    }
    if (mine) {
      if (out_bf16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z, acc.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) = acc;
      }
    }
    if (lane == 0) lse[(long long)h * rows + row] = l_tot;
  }
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// D = dO . O in fp32 per (token, head), plus the log2-domain lse.  A row of
// d elements is read by d * sizeof(T) / 16 lanes with 16-byte loads, so a warp
// covers 32 / that many rows per pass.  Rows are taken in THD order (all heads
// of a token, then the next token), so the reads stream through memory; the
// small D / lse2 writes are the scattered side.
template <typename T>
__device__ __forceinline__ void add_dot16(const T* o, const T* o_lo, const T* g, float& acc) {
  constexpr int kV = 16 / sizeof(T);
  const uint4 a = *reinterpret_cast<const uint4*>(o);
  const uint4 c = *reinterpret_cast<const uint4*>(g);
  uint4 b = make_uint4(0u, 0u, 0u, 0u);
  if (o_lo) b = *reinterpret_cast<const uint4*>(o_lo);
  const T* av = reinterpret_cast<const T*>(&a);
  const T* bv = reinterpret_cast<const T*>(&b);
  const T* cv = reinterpret_cast<const T*>(&c);
#pragma unroll
  for (int i = 0; i < kV; ++i) acc += (to_f(av[i]) + (o_lo ? to_f(bv[i]) : 0.f)) * to_f(cv[i]);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_pre_kernel(const T* __restrict__ o,
                                                           const T* __restrict__ o_lo,
                                                           const T* __restrict__ dout,
                                                           const float* __restrict__ lse, int Tn,
                                                           int H, int d, float* D, float* lse2,
                                                           long long pitch) {
  const int lane = threadIdx.x & 31;
  const int lpr = d * (int)sizeof(T) / 16;          // lanes per row: 8, 16 or 32
  const int rpw = 32 / lpr;                          // rows per warp pass
  const int seg = lane / lpr, sl = lane - seg * lpr;
  const long long pairs = (long long)Tn * H;
  const long long step = (long long)gridDim.x * (kThreads / 32) * rpw;
  for (long long base = ((long long)blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * rpw;
       base < pairs; base += step) {
    const long long w = base + seg;                  // row: token t = w / H, head h
    const bool valid = w < pairs;
    const long long t = valid ? w / H : 0;
    const int h = valid ? (int)(w - t * H) : 0;
    const long long off = (t * H + h) * (long long)d + (long long)sl * (16 / sizeof(T));
    float acc = 0.f;
    if (valid) add_dot16(o + off, o_lo ? o_lo + off : nullptr, dout + off, acc);
    for (int sh = lpr >> 1; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
    if (valid && sl == 0) {
      D[(long long)h * pitch + t] = acc;
      lse2[(long long)h * pitch + t] = lse[(long long)h * Tn + t] * 1.4426950408889634f;
    }
  }
}

// Thread per float4 of the [n*N][H][d] prefix block: fixed-order sum over
// slots 0..n_slots-1 (ranks, then the prefix queries' own term).
__global__ void __launch_bounds__(kThreads) prefix_reduce_kernel(
    const float4* __restrict__ sk, const float4* __restrict__ sv, int n_slots,
    const int32_t* __restrict__ cu, int N, int H, int d, long long pre_rows, float4* dk,
    float4* dv) {
  const long long v_per_row = (long long)H * d / 4;
  const long long total = pre_rows * v_per_row;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const long long prow = x / v_per_row;
    const long long e = x - prow * v_per_row;
    const int i = (int)(prow / N);
    const long long u = prow - (long long)i * N;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int s = 0; s < n_slots; ++s) {
      const float4 ka = sk[(long long)s * total + x];
      const float4 va = sv[(long long)s * total + x];
      a.x += ka.x; a.y += ka.y; a.z += ka.z; a.w += ka.w;
      b.x += va.x; b.y += va.y; b.z += va.z; b.w += va.w;
    }
    const long long nat = ((long long)cu[i] + u) * v_per_row + e;
    dk[nat] = a;
    dv[nat] = b;
  }
}

int grid_for(long long work, int per_block) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (work + per_block - 1) / per_block;
  long long cap = (long long)sms * 8;
  if (want < 1) want = 1;
  return (int)(want < cap ? want : cap);
}

// ---- f16 operand copies -----------------------------------------------------
struct Ptrs4 {
  const uint4* s[4];
  uint4* d[4];
  long long nv[4];   // 16-byte vectors (8 elements) per tensor
};
// member t of a kernel-parameter array, selected without indexing it
// dynamically (which would copy the parameters to local memory)
template <typename T>
__device__ __forceinline__ T pick4(const T (&x)[4], int t) {
  return t == 0 ? x[0] : t == 1 ? x[1] : t == 2 ? x[2] : x[3];
}

// Per block (tensor blockIdx.y): max over |x| of its share, as the bit pattern
// of a non-negative float (bf16 bits shifted into the high half), then one
// atomic max per warp.
__global__ void __launch_bounds__(kThreads) absmax_bf16_kernel(Ptrs4 p, uint32_t* amax) {
  const int t = blockIdx.y;
  const uint4* s = pick4(p.s, t);
  const long long nv = pick4(p.nv, t);
  uint32_t m = 0;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < nv;
       i += (long long)gridDim.x * kThreads) {
    const uint4 v = ld_stream(s + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = max(m, (w[k] & 0x7fffu) << 16);
      m = max(m, w[k] & 0x7fff0000u);
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(&amax[t], m);
}

// Exponent E of max|x| = f * 2^E with f in [0.5, 1) (normal floats), or
// `none` for zero, subnormal or non-finite maxima.
__device__ __forceinline__ int frexp_exp(uint32_t bits, int none) {
  const int biased = (int)(bits >> 23);
  if (biased == 0 || biased == 255) return none;
  return biased - 126;
}
__device__ __forceinline__ int clamp_e(int e) { return e < -60 ? -60 : (e > 60 ? 60 : e); }
// 2^k for |k| <= 126, exactly
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }
// copy exponent of a tensor: its largest magnitude * 2^-e lies in [2^14, 2^15)
__device__ __forceinline__ int copy_e(uint32_t amax_bits) {
  return clamp_e(frexp_exp(amax_bits, 15) - 15);
}

__global__ void __launch_bounds__(kThreads) to_f16_scaled_kernel(Ptrs4 p, OpScales* sc,
                                                                 int backward, int d_log2) {
  const int t = blockIdx.y;
  const int e = copy_e(t == 0 ? sc->amax[0] : sc->amax[1]);
  const float f = pow2i(-e);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (!backward) {
      sc->e[0] = e;
      sc->v_mul = pow2i(e);
    } else {
      const int eq = copy_e(sc->amax[0]), ek = copy_e(sc->amax[1]);
      // |dS| = |P (dP - D)| <= 2 d max|V| max|dO| < 2^(1 + log2 d + E_V + E_dO)
      const int es = clamp_e(1 + d_log2 + frexp_exp(sc->amax[2], 0) +
                             frexp_exp(sc->amax[3], 0) - 15);
      sc->e[0] = eq;
      sc->e[1] = ek;
      sc->qk_mul = pow2i(eq + ek);
      sc->ds_inv = pow2i(-es);
      sc->dq_mul = pow2i(es + ek);
      sc->dk_mul = pow2i(es + eq);
    }
  }
  const uint4* s = pick4(p.s, t);
  uint4* dst = pick4(p.d, t);
  const long long nv = pick4(p.nv, t);
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < nv;
       i += (long long)gridDim.x * kThreads) {
    const uint4 v = ld_stream(s + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16) * f;
      const float hi = __uint_as_float(w[k] & 0xffff0000u) * f;
      const __half2 h = __floats2half2_rn(lo, hi);
      o[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_absmax_bf16(const void* const* src, const int64_t* n, int n_tensors,
                               OpScales* sc, cudaStream_t st) {
  if (n_tensors < 1 || n_tensors > 4) return cudaErrorInvalidValue;
  Ptrs4 p{};
  long long most = 0;
  for (int t = 0; t < n_tensors; ++t) {
    if (n[t] % 8 != 0) return cudaErrorInvalidValue;
    p.s[t] = static_cast<const uint4*>(src[t]);
    p.nv[t] = n[t] / 8;
    most = p.nv[t] > most ? p.nv[t] : most;
  }
  if (most == 0) return cudaSuccess;
  absmax_bf16_kernel<<<dim3(grid_for(most, kThreads), n_tensors), kThreads, 0, st>>>(p, sc->amax);
  return cudaGetLastError();
}

cudaError_t launch_to_f16_scaled(const void* const* src, void* const* dst, const int64_t* n,
                                 int n_tensors, OpScales* sc, bool backward, int d,
                                 cudaStream_t st) {
  if (n_tensors < 1 || n_tensors > 2) return cudaErrorInvalidValue;
  int d_log2 = 0;
  while ((1 << d_log2) < d) ++d_log2;
  Ptrs4 p{};
  long long most = 0;
  for (int t = 0; t < n_tensors; ++t) {
    if (n[t] % 8 != 0) return cudaErrorInvalidValue;
    p.s[t] = static_cast<const uint4*>(src[t]);
    p.d[t] = static_cast<uint4*>(dst[t]);
    p.nv[t] = n[t] / 8;
    most = p.nv[t] > most ? p.nv[t] : most;
  }
  // one block at least: block (0, 0) writes the factors
  to_f16_scaled_kernel<<<dim3(grid_for(most, kThreads), n_tensors), kThreads, 0, st>>>(
      p, sc, backward ? 1 : 0, d_log2);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* const* src, void* const* dst, int n_tensors,
                               size_t row_bytes, const int32_t* idx, int n_rows, bool scatter,
                               cudaStream_t st) {
  if (n_rows <= 0 || n_tensors <= 0) return cudaSuccess;
  RowPtrs p{};
  const uint4** s[4] = {&p.s0, &p.s1, &p.s2, &p.s3};
  uint4** d[4] = {&p.d0, &p.d1, &p.d2, &p.d3};
  for (int i = 0; i < n_tensors && i < 4; ++i) {
    *s[i] = static_cast<const uint4*>(src[i]);
    *d[i] = static_cast<uint4*>(dst[i]);
  }
  const long long warps = (long long)n_rows * n_tensors;
  gather_rows_kernel<<<grid_for(warps, kThreads / 32), kThreads, 0, st>>>(
      p, n_tensors, (int)(row_bytes / 16), idx, n_rows, scatter ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_zigzag_index(const int32_t* smp, int n_seqs, int P, int64_t R,
                                int32_t* fwd_idx, int32_t* inv_idx, cudaStream_t st) {
  if (R == 0 || P < 1) return cudaSuccess;
  // one launch per batch of up to kZigzagBatch samples: each covers, on every
  // rank, the contiguous rank-local rows of its samples
  for (int i0 = 0; i0 < n_seqs; i0 += kZigzagBatch) {
    const int i1 = n_seqs - i0 < kZigzagBatch ? n_seqs : i0 + kZigzagBatch;
    ZigzagBatch b;
    b.n = i1 - i0;
    b.P = P;
    b.R = R;
    b.loc0 = smp[i0 * 4 + 2];
    const long long end = (long long)smp[(i1 - 1) * 4 + 2] + 2LL * smp[(i1 - 1) * 4 + 1];
    b.span = end - b.loc0;
    if (b.span == 0) continue;
    for (int i = i0; i < i1; ++i)
      for (int f = 0; f < 4; ++f) b.smp[i - i0][f] = smp[i * 4 + f];
    const long long n = b.span * (long long)P;
    zigzag_index_kernel<<<grid_for(n, kThreads), kThreads, 0, st>>>(b, fwd_idx, inv_idx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_lse_merge(int n_parts, const float* po, const float* pl, int rows, int H,
                             int d, void* out, bool out_bf16, float* lse, cudaStream_t st) {
  const long long pairs = (long long)rows * H;
  if (pairs == 0) return cudaSuccess;
  if (d % 4 == 0 && d <= 128)
    lse_merge_v4_kernel<<<grid_for(pairs, kThreads / 32), kThreads, 0, st>>>(
        n_parts, po, pl, rows, H, d, out, out_bf16 ? 1 : 0, lse);
  else
    lse_merge_kernel<<<grid_for(pairs, kThreads / 32), kThreads, 0, st>>>(
        n_parts, po, pl, rows, H, d, out, out_bf16 ? 1 : 0, lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const void* out, const void* out_lo, const void* dout, bool bf16,
                                  const float* lse, int T, int H, int d, float* D, float* lse2,
                                  int64_t pitch, cudaStream_t st) {
  const long long pairs = (long long)T * H;
  if (pairs == 0) return cudaSuccess;
  const int g = grid_for((pairs + 3) / 4, kThreads / 32);
  if (bf16)
    bwd_pre_kernel<__nv_bfloat16><<<g, kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(out_lo),
        static_cast<const __nv_bfloat16*>(dout), lse, T,
        H, d, D, lse2, pitch);
  else
    bwd_pre_kernel<float><<<g, kThreads, 0, st>>>(static_cast<const float*>(out), nullptr,
                                                  static_cast<const float*>(dout), lse, T, H, d,
                                                  D, lse2, pitch);
  return cudaGetLastError();
}

cudaError_t launch_prefix_reduce(const float* sk, const float* sv, int n_slots, const int32_t* cu,
                                 int n_seqs, int N, int H, int d, float* dk, float* dv,
                                 cudaStream_t st) {
  const long long pre_rows = (long long)n_seqs * N;
  const long long total = pre_rows * H * d / 4;
  if (total == 0) return cudaSuccess;
  prefix_reduce_kernel<<<grid_for(total, kThreads), kThreads, 0, st>>>(
      reinterpret_cast<const float4*>(sk), reinterpret_cast<const float4*>(sv), n_slots, cu, N, H,
      d, pre_rows, reinterpret_cast<float4*>(dk), reinterpret_cast<float4*>(dv));
  return cudaGetLastError();
}

}  // namespace cpattn
