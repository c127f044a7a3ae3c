// cp_attn_fwd_noalloc: the forward for callers that cannot allocate device
// memory.  Its scratch (work lists, zigzag table, rank-local q/k/v, and for
// fp32 inputs the running result) lives in one fixed array compiled into this
// library instead of a caller-supplied workspace; its status word is the first
// thing in that array.  Host-side uploads are plain copies from the
// plan's own vectors; nothing here calls cudaMalloc, cudaFree, cudaHostAlloc
// or any other allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/cpattn.h"
#include "kernels.h"
#include "plan.h"
#include "tc.h"

namespace cpattn {
void set_last_error(const std::string& msg);
long long device_wait_limit();
}  // namespace cpattn

using namespace cpattn;

namespace {

// The fixed scratch: every GPU that loads the library holds it until exit.
constexpr size_t kScratchBytes = 64ull << 20;
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

cp_status_t fail(cp_status_t s, const std::string& m) {
  set_last_error(m);
  return s;
}

inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of the scratch on the current device (looked up once per
// device, with that device current).
cp_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(CP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(CP_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return fail(CP_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CP_OK;
}

}  // namespace

namespace cpattn {
// Status words of the fixed scratch on the current device, read after the
// caller has synchronised the stream (cp_workspace_status with a NULL
// workspace).  Reads the symbol directly: no allocation.
cudaError_t noalloc_read_status(int32_t out[2]) {
  return cudaMemcpyFromSymbol(out, g_scratch, 2 * sizeof(int32_t), 0, cudaMemcpyDeviceToHost);
}
}  // namespace cpattn

extern "C" cp_status_t cp_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                           cp_dtype_t dt, int T, int H, int d,
                                           const int32_t* cu, int n_seqs, int P, int N,
                                           float scale, void* out, float* lse, void* out_lo,
                                           void* stream) {
  if (dt != CP_F32 && dt != CP_BF16) return fail(CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  if (T < 0 || H < 1 || n_seqs < 1 || P < 1 || N < 0 || !cu)
    return fail(CP_ERR_INVALID_ARG, "T >= 0, H >= 1, n_seqs >= 1, P >= 1, prefix_len >= 0, cu");
  if (d != 64 && d != 128) return fail(CP_ERR_SHAPE, "head_dim must be 64 or 128");
  if (!std::isfinite(scale)) return fail(CP_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (out_lo && dt != CP_BF16) return fail(CP_ERR_DTYPE, "out_lo is for bf16 outputs only");
  const void* ptrs[6] = {q, k, v, out, lse, out_lo};
  for (int i = 0; i < 6 && T > 0; ++i) {
    if (!ptrs[i] && i < 5) return fail(CP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u))
      return fail(CP_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  }
  Problem pb;
  std::string err = make_problem(cu, n_seqs, N, P, T, &pb);
  if (!err.empty()) return fail(CP_ERR_SHAPE, err);
  if (T == 0) return CP_OK;
  const bool bf16 = dt == CP_BF16;
  // bf16: the all-steps tensor-core forward (every ring step of a query tile
  // in one persistent launch, no fp32 running result); fp32: one CUDA-core
  // launch per ring step with the running result in the scratch
  FwdPlan plan;
  plan_forward(pb, true, &plan, bf16 ? kFwdPairQ : kFwdTileQ);
  FusedFwdPlan fused;
  std::vector<int32_t> units, cta_off;
  int sms = 0, grid = 0;
  if (bf16) {
    plan_forward_fused(plan, P, &fused);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long n_units = (long long)fused.items.size() * H;
    if (n_units > 0x7fffffffLL) return fail(CP_ERR_INVALID_ARG, "too many work units");
    grid = (int)fwd_grid(n_units, sms > 0 ? sms : 1);
    if (grid < n_units) plan_unit_lists(fused.items, H, grid, &units, &cta_off);
  }
  std::vector<int32_t> samples;
  int64_t ord = 0;
  for (int i = 0; i < n_seqs; ++i) {
    samples.insert(samples.end(), {pb.cu[i] + N, pb.c[i], pb.off[i], (int32_t)ord});
    ord += 2LL * P * pb.c[i];
  }
  // layout inside the fixed scratch
  const size_t elem = bf16 ? 2 : 4;
  size_t o = 0;
  const size_t o_status = o; o += kStatusBytes;
  const size_t n_items = bf16 ? fused.items.size() : plan.items.size();
  const size_t o_items = o; o = up256(o + n_items * sizeof(FwdItem));
  const size_t o_runs = o; o = up256(o + fused.runs.size() * sizeof(Seg));
  const size_t o_units = o; o = up256(o + (units.size() + cta_off.size()) * sizeof(int32_t));
  const size_t o_idx = o; o = up256(o + (size_t)pb.text_rows * sizeof(int32_t));
  size_t o_qkv[3];
  for (int i = 0; i < 3; ++i) { o_qkv[i] = o; o = up256(o + (size_t)pb.text_rows * H * d * elem); }
  const size_t o_run = o;
  if (!bf16) o = up256(o + (size_t)pb.text_rows * H * d * sizeof(float));
  const size_t o_lrun = o;
  if (!bf16) o = up256(o + (size_t)pb.text_rows * H * sizeof(float));
  // above softmax scale 0.25 the bf16 forward's PV takes an f16 copy of V
  const bool f16 = bf16 && uses_f16_operands(scale);
  const size_t o_scales = o;
  if (f16) o = up256(o + sizeof(OpScales));
  const size_t o_v16 = o;
  if (f16) o = up256(o + (size_t)T * H * d * 2);
  if (o > kScratchBytes) {
    char buf[160];
    snprintf(buf, sizeof buf,
             "this problem needs %zu bytes of scratch; the fixed scratch holds %zu (use cp_attn_fwd "
             "with a workspace)", o, kScratchBytes);
    return fail(CP_ERR_WORKSPACE, buf);
  }
  if (bf16) {
    int dev = 0, major = 0, minor = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(CP_ERR_UNSUPPORTED, "the bf16 path is built for sm_103a (compute capability 10.3)");
  }
  void* base = nullptr;
  cp_status_t s = scratch_address(&base);
  if (s != CP_OK) return s;
  char* w = static_cast<char*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define NA_CUDA(call, what)                                                              \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) return fail(CP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e_)); \
  } while (0)
  // The host arrays below are pageable, so each copy returns only once the
  // source has been read: they may go out of scope when this call returns.
  // The status word must start at zero; everything else is written before it
  // is read.
  NA_CUDA(cudaMemsetAsync(w + o_status, 0, kStatusBytes, st), "clear status");
  const void* items_src = bf16 ? (const void*)fused.items.data() : (const void*)plan.items.data();
  NA_CUDA(cudaMemcpyAsync(w + o_items, items_src, n_items * sizeof(FwdItem),
                          cudaMemcpyHostToDevice, st),
          "upload work list");
  if (!fused.runs.empty())
    NA_CUDA(cudaMemcpyAsync(w + o_runs, fused.runs.data(), fused.runs.size() * sizeof(Seg),
                            cudaMemcpyHostToDevice, st),
            "upload key runs");
  if (!units.empty()) {
    NA_CUDA(cudaMemcpyAsync(w + o_units, units.data(), units.size() * sizeof(int32_t),
                            cudaMemcpyHostToDevice, st),
            "upload unit lists");
    NA_CUDA(cudaMemcpyAsync(w + o_units + units.size() * sizeof(int32_t), cta_off.data(),
                            cta_off.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st),
            "upload unit list offsets");
  }
  int32_t* idx = reinterpret_cast<int32_t*>(w + o_idx);
  NA_CUDA(launch_zigzag_index(samples.data(), n_seqs, P, pb.R, idx, nullptr, st),
          "zigzag index kernel");
  OpScales* sc = reinterpret_cast<OpScales*>(w + o_scales);
  const void* vsrc = v;
  if (f16) {
    const int64_t n = (int64_t)T * H * d;
    void* v16 = w + o_v16;
    NA_CUDA(cudaMemsetAsync(sc, 0, sizeof(OpScales), st), "clear operand scales");
    NA_CUDA(launch_absmax_bf16(&v, &n, 1, sc, st), "max |V|");
    NA_CUDA(launch_to_f16_scaled(&v, &v16, &n, 1, sc, false, d, st), "f16 copy of V");
    vsrc = v16;
  }
  const void* src[3] = {q, k, vsrc};
  void* dst[3] = {w + o_qkv[0], w + o_qkv[1], w + o_qkv[2]};
  NA_CUDA(launch_gather_rows(src, dst, 3, (size_t)H * d * elem, idx, (int)pb.text_rows, false, st),
          "zigzag gather");
  const FwdItem* items = reinterpret_cast<const FwdItem*>(w + o_items);
  if (bf16) {
    TcFwdArgs a;
    const char* terr = nullptr;
    const int64_t PR = pb.text_rows;
    const bool ok = make_tmap_thd(&a.tm_q_text, dst[0], PR, H, d, 128, &terr) &&
                    make_tmap_thd(&a.tm_k_text, dst[1], PR, H, d, 128, &terr) &&
                    make_tmap_thd(&a.tm_v_text, dst[2], PR, H, d, 128, &terr, f16) &&
                    make_tmap_thd(&a.tm_q_nat, q, T, H, d, 128, &terr) &&
                    make_tmap_thd(&a.tm_k_nat, k, T, H, d, 128, &terr) &&
                    make_tmap_thd(&a.tm_v_nat, vsrc, T, H, d, 128, &terr, f16);
    if (!ok) return fail(CP_ERR_CUDA, std::string("tensor map: ") + (terr ? terr : "?"));
    a.H = H; a.Hkv = H; a.d = d; a.pdl = 0;
    a.items = items;
    a.n_items = (int)fused.items.size();
    a.runs = reinterpret_cast<const Seg*>(w + o_runs);
    a.units = nullptr;
    a.cta_off = nullptr;
    a.n_ctas = 0;
    if (!units.empty()) {
      a.units = reinterpret_cast<const int32_t*>(w + o_units);
      a.cta_off = a.units + units.size();
      a.n_ctas = grid;
    }
    a.scale_log2 = scale * 1.4426950408889634f;
    a.f16_pv = f16 ? 1 : 0;
    a.op_scales = f16 ? sc : nullptr;
    a.o_run = nullptr; a.lse_run = nullptr; a.run_rows = 0;
    a.text_rows = PR;
    a.out = out; a.lse = lse; a.T = T; a.out_lo = out_lo;
    a.status = reinterpret_cast<int32_t*>(w + o_status);
    a.wait_limit = device_wait_limit();
    NA_CUDA(launch_tc_fwd(a, st), "tensor-core forward (all ring steps)");
    return CP_OK;
  }
  SimtFwdArgs a;
  a.q_text = dst[0]; a.k_text = dst[1]; a.v_text = dst[2];
  a.q_nat = q; a.k_nat = k; a.v_nat = v;
  a.H = H; a.Hkv = H; a.d = d; a.scale = scale;
  a.o_run = reinterpret_cast<float*>(w + o_run);
  a.lse_run = reinterpret_cast<float*>(w + o_lrun);
  a.run_rows = pb.text_rows;
  a.out = out; a.lse = lse; a.T = T;
  for (int step = 0; step < P; ++step) {
    a.items = items + plan.step_begin[step];
    a.n_items = plan.step_begin[step + 1] - plan.step_begin[step];
    NA_CUDA(launch_simt_fwd(a, st), "ring step");
  }
#undef NA_CUDA
  return CP_OK;
}
