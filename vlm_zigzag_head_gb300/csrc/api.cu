// C ABI of libcpattn: argument checks, work-list planning and upload,
// workspace layout, and the launch sequence of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/cpattn.h"
#include "check.cuh"
#include "kernels.h"
#include "plan.h"
#include "tc.h"

using namespace cpattn;

namespace {

thread_local std::string g_err;
std::atomic<long long> g_wait_limit{0};

cp_status_t fail(cp_status_t s, const std::string& msg) {
  g_err = msg;
  return s;
}

cp_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(CP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CP_CUDA(call, what)                        \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// page-locked staging ring: work lists are copied host -> device without the
// implicit stream synchronisation of pageable copies.  A slot is reused only
// after the event recorded behind its last copy has completed.
// ---------------------------------------------------------------------------
class Stager {
 public:
  cudaError_t upload(void* dst, const void* src, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu_);
    Slot& s = slots_[next_];
    next_ = (next_ + 1) % kSlots;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (s.ev && s.used) {
      e = cudaEventSynchronize(s.ev);
      if (e != cudaSuccess) return e;
    }
    if (s.ev && s.dev != dev) {
      cudaEventDestroy(s.ev);
      s.ev = nullptr;
    }
    if (!s.ev) {
      e = cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
      s.dev = dev;
    }
    if (s.cap < bytes) {
      if (s.host) cudaFreeHost(s.host);
      s.host = nullptr;
      s.cap = 0;
      size_t cap = align_up(bytes * 2, 1 << 16);
      e = cudaHostAlloc(&s.host, cap, cudaHostAllocDefault);
      if (e != cudaSuccess) return e;
      s.cap = cap;
    }
    memcpy(s.host, src, bytes);
    e = cudaMemcpyAsync(dst, s.host, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(s.ev, st);
    s.used = (e == cudaSuccess);
    return e;
  }

 private:
  static constexpr int kSlots = 16;
  struct Slot {
    void* host = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    int dev = -1;
    bool used = false;
  };
  std::mutex mu_;
  Slot slots_[kSlots];
  int next_ = 0;
};

Stager& stager() {
  static Stager* s = new Stager();  // intentionally leaked: outlives static destructors
  return *s;
}

// ---------------------------------------------------------------------------
// plan cache (plans depend only on cu_seqlens, prefix_len and P)
// ---------------------------------------------------------------------------
// Unit lists of the persistent all-steps forward for one (heads, grid):
// `packed` holds the units, then cta_off (grid + 1 entries).
struct UnitLists {
  int H = 0, grid = 0;
  size_t n_units = 0;
  std::vector<int32_t> packed;
};

struct PlanSet {
  Problem pb;
  FwdPlan fwd;       // text rows in rank-local order, 128-row items (CUDA cores)
  FwdPlan fwd2;      // text rows in rank-local order, 256-row items (tensor cores)
  FusedFwdPlan fused;  // fwd2 with all ring steps of a query tile in one item
  FwdPlan fwd_nat;   // text rows in natural order (fp32 dQ pass)
  BwdPlan bwd;
  FusedBwdPlan bwd_fused;   // bwd with all ring steps of a key tile in one item (128-query kernel)
  FusedBwdPlan bwd_fused_merged;   // the same with each prefix key tile's slots in one item
  std::vector<int32_t> samples;  // [n][4]: t0, c, off, ord0 (index kernel)
  std::mutex ul_mu;
  std::vector<std::shared_ptr<const UnitLists>> ul;  // recent unit lists
};

std::shared_ptr<const UnitLists> unit_lists(PlanSet& ps, int H, int grid) {
  std::lock_guard<std::mutex> lk(ps.ul_mu);
  for (const auto& p : ps.ul)
    if (p->H == H && p->grid == grid) return p;
  auto u = std::make_shared<UnitLists>();
  u->H = H;
  u->grid = grid;
  std::vector<int32_t> cta_off;
  plan_unit_lists(ps.fused.items, H, grid, &u->packed, &cta_off);
  u->n_units = u->packed.size();
  u->packed.insert(u->packed.end(), cta_off.begin(), cta_off.end());
  ps.ul.push_back(u);
  if (ps.ul.size() > 4) ps.ul.erase(ps.ul.begin());
  return u;
}

struct PlanCache {
  std::mutex mu;
  std::vector<std::shared_ptr<PlanSet>> lru;
};

PlanCache& plan_cache() {
  static PlanCache* c = new PlanCache();
  return *c;
}

cp_status_t get_plans(const int32_t* cu, int n_seqs, int N, int P, int T, int H, int d,
                      std::shared_ptr<PlanSet>* out) {
  Problem pb;
  std::string err = make_problem(cu, n_seqs, N, P, T, &pb);
  if (!err.empty()) return fail(CP_ERR_SHAPE, err);
  PlanCache& pc = plan_cache();
  {
    std::lock_guard<std::mutex> lk(pc.mu);
    for (auto& p : pc.lru) {
      if (p->pb.P == P && p->pb.N == N && p->pb.cu == pb.cu) {
        *out = p;
        return CP_OK;
      }
    }
  }
  auto ps = std::make_shared<PlanSet>();
  ps->pb = pb;
  plan_forward(pb, true, &ps->fwd);
  plan_forward(pb, true, &ps->fwd2, kFwdPairQ);
  plan_forward_fused(ps->fwd2, P, &ps->fused);
  plan_forward(pb, false, &ps->fwd_nat);
  plan_backward(pb, &ps->bwd);
  plan_backward_fused(ps->bwd, P, 128, false, &ps->bwd_fused);
  plan_backward_fused(ps->bwd, P, 128, true, &ps->bwd_fused_merged);
  int64_t ord = 0;
  for (int i = 0; i < n_seqs; ++i) {
    ps->samples.push_back(pb.cu[i] + N);
    ps->samples.push_back(pb.c[i]);
    ps->samples.push_back(pb.off[i]);
    ps->samples.push_back((int32_t)ord);
    ord += 2LL * P * pb.c[i];
  }
  std::lock_guard<std::mutex> lk(pc.mu);
  pc.lru.insert(pc.lru.begin(), ps);
  if (pc.lru.size() > 8) pc.lru.pop_back();
  *out = ps;
  return CP_OK;
}

// ---------------------------------------------------------------------------
// workspace layouts
// ---------------------------------------------------------------------------
struct FwdWs {
  size_t status = 0, items = 0, runs = 0, units = 0, idx = 0, qkv[3] = {0, 0, 0},
         o_run = 0, lse_run = 0, scales = 0, v16 = 0, total = 0;
};

// `running`: reserve the fp32 running result (o_run, lse_run) that the
// per-step schedules merge into (fp32 inputs, or bf16 under
// CPATTN_FWD_PER_STEP=1).  The default all-steps tensor-core forward keeps its
// merge on chip and needs none.
// `f16`: the f16 copy of V and its factors (bf16 above softmax scale 0.25).
FwdWs fwd_layout(const PlanSet& ps, int H, int Hkv, int d, size_t elem, bool running, bool f16) {
  FwdWs w;
  size_t o = 0;
  w.status = o; o += kStatusBytes;
  w.items = o;
  o = align_up(o + std::max(ps.fwd.items.size(), ps.fused.items.size()) * sizeof(FwdItem), 256);
  w.runs = o; o = align_up(o + ps.fused.runs.size() * sizeof(Seg), 256);
  // unit lists: units, then cta_off (at most units + 1 entries)
  w.units = o; o = align_up(o + (2 * ps.fused.items.size() * H + 1) * sizeof(int32_t), 256);
  w.idx = o; o = align_up(o + (size_t)ps.pb.text_rows * sizeof(int32_t), 256);
  // rank-local q [rows][H][d]; k, v [rows][Hkv][d]
  for (int i = 0; i < 3; ++i) {
    w.qkv[i] = o;
    o = align_up(o + (size_t)ps.pb.text_rows * (i == 0 ? H : Hkv) * d * elem, 256);
  }
  w.o_run = o;
  if (running) o = align_up(o + (size_t)ps.pb.text_rows * H * d * sizeof(float), 256);
  w.lse_run = o;
  if (running) o = align_up(o + (size_t)ps.pb.text_rows * H * sizeof(float), 256);
  w.scales = o;
  if (f16) o = align_up(o + sizeof(OpScales), 256);
  w.v16 = o;
  if (f16) o = align_up(o + (size_t)ps.pb.T * Hkv * d * 2, 256);
  w.total = o;
  return w;
}

struct BwdWs {
  size_t status = 0, items = 0, runs = 0, qitems = 0, cu = 0, D = 0, lse2 = 0, slots = 0,
         scales = 0, q16 = 0, k16 = 0, total = 0;
};

inline int64_t ld_pitch(int64_t T) { return (T + 3) / 4 * 4; }

// `f16`: the f16 copies of Q and K and their factors (bf16 above softmax
// scale 0.25).
BwdWs bwd_layout(const PlanSet& ps, int H, int Hkv, int d, bool simt, bool own_slots, bool f16) {
  BwdWs w;
  const Problem& pb = ps.pb;
  size_t o = 0;
  w.status = o; o += kStatusBytes;
  w.items = o;
  o = align_up(o + std::max(ps.bwd.items.size(), ps.bwd_fused.items.size()) * sizeof(BwdItem), 256);
  w.runs = o;
  if (!simt)
    o = align_up(o + std::max(ps.bwd_fused.runs.size(), ps.bwd_fused_merged.runs.size()) *
                         sizeof(Seg), 256);
  w.qitems = o;
  if (simt) o = align_up(o + ps.fwd_nat.items.size() * sizeof(FwdItem), 256);
  w.cu = o; o = align_up(o + pb.cu.size() * sizeof(int32_t), 256);
  // lse2 and D planes [2][H][pitch], pitch = T rounded up to 4 (16-byte rows for TMA)
  w.lse2 = o;
  w.D = o + (size_t)ld_pitch(pb.T) * H * sizeof(float);  // plane 1 directly after plane 0
  o = align_up(o + 2 * (size_t)ld_pitch(pb.T) * H * sizeof(float), 256);
  w.slots = o;
  if (own_slots)
    o = align_up(o + 2ull * (pb.P + 1) * pb.n_seqs * pb.N * Hkv * d * sizeof(float), 256);
  w.scales = o;
  if (f16) o = align_up(o + sizeof(OpScales), 256);
  w.q16 = o;
  if (f16) o = align_up(o + (size_t)pb.T * H * d * 2, 256);
  w.k16 = o;
  if (f16) o = align_up(o + (size_t)pb.T * Hkv * d * 2, 256);
  w.total = o;
  return w;
}

cp_status_t check_common(const void* const* ptrs, int n_ptrs, cp_dtype_t dt, int T, int H,
                         int Hkv, int d, const int32_t* cu, int n_seqs, int P, int N,
                         float scale) {
  if (dt != CP_F32 && dt != CP_BF16) return fail(CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  if (T < 0 || H < 1 || n_seqs < 1 || P < 1 || N < 0)
    return fail(CP_ERR_INVALID_ARG, "T >= 0, H >= 1, n_seqs >= 1, P >= 1, prefix_len >= 0");
  if (Hkv < 1 || H % Hkv != 0)
    return fail(CP_ERR_SHAPE, "H must be a positive multiple of H_kv");
  if (!cu) return fail(CP_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (d != 64 && d != 128) return fail(CP_ERR_SHAPE, "head_dim must be 64 or 128");
  if (!std::isfinite(scale)) return fail(CP_ERR_INVALID_ARG, "softmax_scale must be finite");
  for (int i = 0; i < n_ptrs && T > 0; ++i) {
    if (!ptrs[i]) return fail(CP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned16(ptrs[i])) return fail(CP_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  }
  return CP_OK;
}

cp_status_t check_device_for_bf16() {
  int dev = 0, major = 0, minor = 0;
  CP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  CP_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cc major");
  CP_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cc minor");
  if (major != 10 || minor != 3)
    return fail(CP_ERR_UNSUPPORTED, "the bf16 path is built for sm_103a (compute capability 10.3)");
  return CP_OK;
}

// The tensor-core forward runs all ring steps in one launch unless
// CPATTN_FWD_PER_STEP=1 asks for one launch per ring step with the fp32
// running result in between (the same arithmetic, merged in another order).
bool use_fused_forward() {
  static int v = [] {
    const char* e = getenv("CPATTN_FWD_PER_STEP");
    return (e && e[0] == '1') ? 0 : 1;
  }();
  return v != 0;
}

// The forward of this dtype merges ring steps through the fp32 running result.
bool fwd_needs_running(cp_dtype_t dt) { return dt != CP_BF16 || !use_fused_forward(); }

long long wait_limit() {
  long long w = g_wait_limit.load();
  return w > 0 ? w : (1LL << 22);
}

// ---------------------------------------------------------------------------
// optional per-launch timing: CUDA events recorded on the launching stream
// around every kernel of the path while profiling is on
// ---------------------------------------------------------------------------
constexpr int kProfKinds = 8;
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
  int count;   // launches between the two events
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<ProfRec> g_prof;

struct ProfScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  int count;
  ProfScope(int k, cudaStream_t s, int n = 1) : kind(k), st(s), count(n) {
    if (!g_prof_on.load()) return;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
      a = b = nullptr;
      return;
    }
    cudaEventRecord(a, st);
  }
  ~ProfScope() {
    if (!a) return;
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({kind, a, b, count});
  }
};

}  // namespace

namespace cpattn {
cudaError_t noalloc_read_status(int32_t out[2]);   // noalloc.cu
// Shared with other translation units of the library (the fixed-scratch entry
// point): the thread-local error message and the device wait bound.
void set_last_error(const std::string& msg) { g_err = msg; }
long long device_wait_limit() { return wait_limit(); }
}  // namespace cpattn

extern "C" {

const char* cp_last_error(void) { return g_err.c_str(); }

const char* cp_status_string(cp_status_t s) {
  switch (s) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_SHAPE: return "CP_ERR_SHAPE";
    case CP_ERR_DTYPE: return "CP_ERR_DTYPE";
    case CP_ERR_ALIGNMENT: return "CP_ERR_ALIGNMENT";
    case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_BOUNDS: return "CP_ERR_BOUNDS";
  }
  return "CP_ERR_UNKNOWN";
}

int cp_version(void) { return CPATTN_VERSION; }

void cp_set_wait_limit(long long rounds) { g_wait_limit.store(rounds > 0 ? rounds : 0); }

cp_status_t cp_zigzag_index(const int32_t* cu, int n_seqs, int N, int P, int32_t* fwd_idx,
                            int32_t* inv_idx, int on_device, void* stream) {
  if (!cu || n_seqs < 1 || P < 1 || N < 0)
    return fail(CP_ERR_INVALID_ARG, "cu_seqlens non-NULL, n_seqs >= 1, P >= 1, prefix_len >= 0");
  if (on_device) {
    std::shared_ptr<PlanSet> ps;
    cp_status_t s = get_plans(cu, n_seqs, N, P, -1, 1, 64, &ps);
    if (s != CP_OK) return s;
    if ((fwd_idx && !aligned16(fwd_idx)) || (inv_idx && !aligned16(inv_idx)))
      return fail(CP_ERR_ALIGNMENT, "index tables must be 16-byte aligned");
    if (ps->pb.text_rows == 0 || (!fwd_idx && !inv_idx)) return CP_OK;
    // the device kernel cp_attn_fwd runs for its own table
    ProfScope ps_(0, static_cast<cudaStream_t>(stream));
    CP_CUDA(launch_zigzag_index(ps->samples.data(), n_seqs, P, ps->pb.R, fwd_idx, inv_idx,
                                static_cast<cudaStream_t>(stream)),
            "zigzag index kernel");
    return CP_OK;
  }
  Problem pb;
  std::string err = make_problem(cu, n_seqs, N, P, -1, &pb);
  if (!err.empty()) return fail(CP_ERR_SHAPE, err);
  zigzag_tables(pb, fwd_idx, inv_idx);
  return CP_OK;
}

cp_status_t cp_zigzag_gather(const void* src, void* dst, size_t row_bytes, const int32_t* idx,
                             int n_rows, void* stream) {
  if (n_rows < 0) return fail(CP_ERR_INVALID_ARG, "n_rows < 0");
  if (n_rows == 0) return CP_OK;
  if (!src || !dst || !idx) return fail(CP_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(dst) || (row_bytes % 16) != 0 || row_bytes == 0)
    return fail(CP_ERR_ALIGNMENT, "pointers and row_bytes must be multiples of 16");
  const void* s[1] = {src};
  void* d[1] = {dst};
  CP_CUDA(launch_gather_rows(s, d, 1, row_bytes, idx, n_rows, false,
                             static_cast<cudaStream_t>(stream)),
          "zigzag gather");
  return CP_OK;
}

cp_status_t cp_zigzag_scatter(const void* src, void* dst, size_t row_bytes, const int32_t* idx,
                              int n_rows, void* stream) {
  if (n_rows < 0) return fail(CP_ERR_INVALID_ARG, "n_rows < 0");
  if (n_rows == 0) return CP_OK;
  if (!src || !dst || !idx) return fail(CP_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(dst) || (row_bytes % 16) != 0 || row_bytes == 0)
    return fail(CP_ERR_ALIGNMENT, "pointers and row_bytes must be multiples of 16");
  const void* s[1] = {src};
  void* d[1] = {dst};
  CP_CUDA(launch_gather_rows(s, d, 1, row_bytes, idx, n_rows, true,
                             static_cast<cudaStream_t>(stream)),
          "zigzag scatter");
  return CP_OK;
}

size_t cp_attn_fwd_workspace_size_gqa(cp_dtype_t dt, int T, int H, int Hkv, int d,
                                      const int32_t* cu, int n_seqs, int P, int N, float scale) {
  std::shared_ptr<PlanSet> ps;
  if (!cu || H < 1 || Hkv < 1 || H % Hkv != 0 || (dt != CP_F32 && dt != CP_BF16)) return 0;
  if (get_plans(cu, n_seqs, N, P, T, H, d, &ps) != CP_OK) return 0;
  const bool f16 = dt == CP_BF16 && uses_f16_operands(scale);
  return fwd_layout(*ps, H, Hkv, d, dt == CP_BF16 ? 2 : 4, fwd_needs_running(dt), f16).total;
}

size_t cp_attn_fwd_workspace_size(cp_dtype_t dt, int T, int H, int d, const int32_t* cu,
                                  int n_seqs, int P, int N, float scale) {
  return cp_attn_fwd_workspace_size_gqa(dt, T, H, H, d, cu, n_seqs, P, N, scale);
}

cp_status_t cp_attn_fwd(const void* q, const void* k, const void* v, cp_dtype_t dt, int T, int H,
                        int d, const int32_t* cu, int n_seqs, int P, int N, float scale,
                        void* out, float* lse, void* out_lo, void* ws, size_t ws_bytes,
                        void* stream) {
  return cp_attn_fwd_gqa(q, k, v, dt, T, H, H, d, cu, n_seqs, P, N, scale, out, lse, out_lo, ws,
                         ws_bytes, stream);
}

cp_status_t cp_attn_fwd_gqa(const void* q, const void* k, const void* v, cp_dtype_t dt, int T,
                            int H, int Hkv, int d, const int32_t* cu, int n_seqs, int P, int N,
                            float scale, void* out, float* lse, void* out_lo, void* ws,
                            size_t ws_bytes, void* stream) {
  const void* ptrs[5] = {q, k, v, out, lse};
  cp_status_t s = check_common(ptrs, 5, dt, T, H, Hkv, d, cu, n_seqs, P, N, scale);
  if (s != CP_OK) return s;
  if (out_lo && dt != CP_BF16) return fail(CP_ERR_DTYPE, "out_lo is for bf16 outputs only");
  if (out_lo && !aligned16(out_lo)) return fail(CP_ERR_ALIGNMENT, "out_lo alignment");
  std::shared_ptr<PlanSet> ps;
  s = get_plans(cu, n_seqs, N, P, T, H, d, &ps);
  if (s != CP_OK) return s;
  if (T == 0) return CP_OK;
  const bool bf16 = dt == CP_BF16;
  const bool tc = bf16;   // bf16: tensor cores; fp32: the CUDA-core parity path
  if (tc && (s = check_device_for_bf16()) != CP_OK) return s;
  const size_t elem = bf16 ? 2 : 4;
  const bool f16 = tc && uses_f16_operands(scale);
  const FwdWs L = fwd_layout(*ps, H, Hkv, d, elem, fwd_needs_running(dt), f16);
  if (!ws || ws_bytes < L.total)
    return fail(CP_ERR_WORKSPACE, "workspace smaller than cp_attn_fwd_workspace_size()");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(CP_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const Problem& pb = ps->pb;
  CP_CUDA(cudaMemsetAsync(w + L.status, 0, kStatusBytes, st), "clear status");
  const FwdPlan& fp = tc ? ps->fwd2 : ps->fwd;  // items of 256 (tensor cores) / 128 rows
  const bool fused = tc && use_fused_forward();
  if (fused) {
    CP_CUDA(stager().upload(w + L.items, ps->fused.items.data(),
                            ps->fused.items.size() * sizeof(FwdItem), st),
            "upload work list");
    CP_CUDA(stager().upload(w + L.runs, ps->fused.runs.data(),
                            ps->fused.runs.size() * sizeof(Seg), st),
            "upload key runs");
  } else {
    CP_CUDA(stager().upload(w + L.items, fp.items.data(), fp.items.size() * sizeof(FwdItem), st),
            "upload work list");
  }
  int32_t* idx = reinterpret_cast<int32_t*>(w + L.idx);
  // get_batch_on_this_cp_rank: zigzag table, then index_select of q, k, v text rows
  {
    ProfScope ps_(0, st);
    CP_CUDA(launch_zigzag_index(ps->samples.data(), n_seqs, P, pb.R, idx, nullptr, st),
            "zigzag index kernel");
  }
  // above softmax scale 0.25: PV on f16 operands, V from its scaled f16 copy
  OpScales* sc = reinterpret_cast<OpScales*>(w + L.scales);
  const void* vsrc = v;
  const void* src[3] = {q, k, v};
  void* dst[3] = {w + L.qkv[0], w + L.qkv[1], w + L.qkv[2]};
  {
    ProfScope ps_(1, st, f16 ? 3 : 1);
    if (f16) {
      const int64_t n = (int64_t)T * Hkv * d;
      void* v16 = w + L.v16;
      CP_CUDA(cudaMemsetAsync(sc, 0, sizeof(OpScales), st), "clear operand scales");
      CP_CUDA(launch_absmax_bf16(&v, &n, 1, sc, st), "max |V|");
      CP_CUDA(launch_to_f16_scaled(&v, &v16, &n, 1, sc, false, d, st), "f16 copy of V");
      vsrc = v16;
      src[2] = vsrc;
    }
    if (Hkv == H) {
      CP_CUDA(launch_gather_rows(src, dst, 3, (size_t)H * d * elem, idx, (int)pb.text_rows,
                                 false, st),
              "zigzag gather");
    } else {  // q rows and the narrower k / v rows
      CP_CUDA(launch_gather_rows(src, dst, 1, (size_t)H * d * elem, idx, (int)pb.text_rows,
                                 false, st),
              "zigzag gather");
      CP_CUDA(launch_gather_rows(src + 1, dst + 1, 2, (size_t)Hkv * d * elem, idx,
                                 (int)pb.text_rows, false, st),
              "zigzag gather");
    }
  }
  const FwdItem* items = reinterpret_cast<const FwdItem*>(w + L.items);
  float* o_run = reinterpret_cast<float*>(w + L.o_run);
  float* lse_run = reinterpret_cast<float*>(w + L.lse_run);
  if (tc) {
    TcFwdArgs a;
    const char* terr = nullptr;
    const int64_t PR = pb.text_rows;
    bool ok = make_tmap_thd(&a.tm_q_text, dst[0], PR, H, d, 128, &terr) &&
              make_tmap_thd(&a.tm_k_text, dst[1], PR, Hkv, d, 128, &terr) &&
              make_tmap_thd(&a.tm_v_text, dst[2], PR, Hkv, d, 128, &terr, f16) &&
              make_tmap_thd(&a.tm_q_nat, q, T, H, d, 128, &terr) &&
              make_tmap_thd(&a.tm_k_nat, k, T, Hkv, d, 128, &terr) &&
              make_tmap_thd(&a.tm_v_nat, vsrc, T, Hkv, d, 128, &terr, f16);
    if (!ok) return fail(CP_ERR_CUDA, std::string("tensor map: ") + (terr ? terr : "?"));
    a.H = H; a.Hkv = Hkv; a.d = d;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.f16_pv = f16 ? 1 : 0;
    a.op_scales = f16 ? sc : nullptr;
    a.o_run = o_run; a.lse_run = lse_run; a.run_rows = PR;
    a.text_rows = PR;
    a.out = out; a.lse = lse; a.T = T; a.out_lo = out_lo;
    a.status = reinterpret_cast<int32_t*>(w + L.status);
    a.wait_limit = wait_limit();
    a.runs = nullptr;
    a.units = nullptr;
    a.cta_off = nullptr;
    a.n_ctas = 0;
    if (fused) {  // every ring step of every query tile in one persistent launch
      a.items = items;
      a.n_items = (int)ps->fused.items.size();
      a.runs = reinterpret_cast<const Seg*>(w + L.runs);
      a.pdl = 0;
      int dev = 0, sms = 0;
      CP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
      CP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
      const long long units = (long long)a.n_items * H;
      const long long grid = fwd_grid(units, sms);
      if (grid < units) {  // persistent CTAs: equal shares of work, head by head
        std::shared_ptr<const UnitLists> ul = unit_lists(*ps, H, (int)grid);
        CP_CUDA(stager().upload(w + L.units, ul->packed.data(),
                                ul->packed.size() * sizeof(int32_t), st),
                "upload unit lists");
        a.units = reinterpret_cast<const int32_t*>(w + L.units);
        a.cta_off = a.units + ul->n_units;
        a.n_ctas = (int)grid;
      }
      ProfScope ps_(2, st);
      CP_CUDA(launch_tc_fwd(a, st), "tensor-core forward (all ring steps)");
      return CP_OK;
    }
    // Ring steps after the first are programmatic dependents of the one
    // before: their CTAs fill SMs as the previous step drains and wait for it
    // only at the merge.  One profiling interval spans the P launches.
    // (Only a step that directly follows a launched step kernel may be a
    // dependent: an empty step launches nothing.)
    ProfScope ps_(2, st, P);
    bool prev = false;
    for (int step = 0; step < P; ++step) {
      a.items = items + fp.step_begin[step];
      a.n_items = fp.step_begin[step + 1] - fp.step_begin[step];
      a.pdl = prev ? 1 : 0;
      CP_CUDA(launch_tc_fwd(a, st), "tensor-core ring step");
      prev = a.n_items > 0;
    }
    return CP_OK;
  }
  SimtFwdArgs a;
  a.q_text = dst[0]; a.k_text = dst[1]; a.v_text = dst[2];
  a.q_nat = q; a.k_nat = k; a.v_nat = v;
  a.H = H; a.Hkv = Hkv; a.d = d; a.scale = scale;
  a.o_run = o_run; a.lse_run = lse_run; a.run_rows = pb.text_rows;
  a.out = out; a.lse = lse; a.T = T;
  for (int step = 0; step < P; ++step) {
    a.items = items + fp.step_begin[step];
    a.n_items = fp.step_begin[step + 1] - fp.step_begin[step];
    ProfScope ps_(6, st);
    CP_CUDA(launch_simt_fwd(a, st), "ring step");
  }
  return CP_OK;
}

cp_status_t cp_copy_rows(void* dst, size_t dst_pitch, const void* src, size_t src_pitch,
                         size_t width, size_t rows, void* stream) {
  if (rows == 0 || width == 0) return CP_OK;
  if (!dst || !src) return fail(CP_ERR_INVALID_ARG, "NULL pointer");
  if (width > dst_pitch || width > src_pitch) return fail(CP_ERR_INVALID_ARG, "width > pitch");
  CP_CUDA(cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, width, rows, cudaMemcpyDefault,
                            static_cast<cudaStream_t>(stream)),
          "strided row copy");
  return CP_OK;
}

cp_status_t cp_lse_merge(int n_parts, const float* part_out, const float* part_lse, int rows,
                         int H, int d, void* out, cp_dtype_t out_dt, float* lse, void* stream) {
  if (n_parts < 1 || rows < 0 || H < 1 || d < 1 || d > 128)
    return fail(CP_ERR_INVALID_ARG, "n_parts >= 1, rows >= 0, H >= 1, 1 <= d <= 128");
  if (out_dt != CP_F32 && out_dt != CP_BF16) return fail(CP_ERR_DTYPE, "out dtype");
  if (rows == 0) return CP_OK;
  const void* ptrs[4] = {part_out, part_lse, out, lse};
  for (const void* p : ptrs) {
    if (!p) return fail(CP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(p)) return fail(CP_ERR_ALIGNMENT, "pointers must be 16-byte aligned");
  }
  CP_CUDA(launch_lse_merge(n_parts, part_out, part_lse, rows, H, d, out, out_dt == CP_BF16, lse,
                           static_cast<cudaStream_t>(stream)),
          "lse merge");
  return CP_OK;
}

size_t cp_attn_bwd_workspace_size_gqa(cp_dtype_t dt, int T, int H, int Hkv, int d,
                                      const int32_t* cu, int n_seqs, int P, int N, float scale) {
  std::shared_ptr<PlanSet> ps;
  if (!cu || H < 1 || Hkv < 1 || H % Hkv != 0 || (dt != CP_F32 && dt != CP_BF16)) return 0;
  if (get_plans(cu, n_seqs, N, P, T, H, d, &ps) != CP_OK) return 0;
  const bool simt = dt != CP_BF16;   // fp32: the CUDA-core parity path
  // per-rank prefix slots in the workspace: only the CUDA-core path needs them
  // when the caller does not ask for them (the tensor-core path then sums the
  // ranks' prefix terms on chip)
  return bwd_layout(*ps, H, Hkv, d, simt, simt, !simt && uses_f16_operands(scale)).total;
}

size_t cp_attn_bwd_workspace_size(cp_dtype_t dt, int T, int H, int d, const int32_t* cu,
                                  int n_seqs, int P, int N, float scale) {
  return cp_attn_bwd_workspace_size_gqa(dt, T, H, H, d, cu, n_seqs, P, N, scale);
}

cp_status_t cp_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const void* out_lo, const float* lse, const void* dout, cp_dtype_t dt,
                        int T, int H, int d,
                        const int32_t* cu, int n_seqs, int P, int N, float scale, float* dq,
                        float* dk, float* dv, float* pgrad, void* ws, size_t ws_bytes,
                        void* stream) {
  return cp_attn_bwd_gqa(q, k, v, out, out_lo, lse, dout, dt, T, H, H, d, cu, n_seqs, P, N,
                         scale, dq, dk, dv, pgrad, ws, ws_bytes, stream);
}

cp_status_t cp_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* out,
                            const void* out_lo, const float* lse, const void* dout,
                            cp_dtype_t dt, int T, int H, int Hkv, int d, const int32_t* cu,
                            int n_seqs, int P, int N, float scale, float* dq, float* dk,
                            float* dv, float* pgrad, void* ws, size_t ws_bytes, void* stream) {
  const void* ptrs[9] = {q, k, v, out, lse, dout, dq, dk, dv};
  cp_status_t s = check_common(ptrs, 9, dt, T, H, Hkv, d, cu, n_seqs, P, N, scale);
  if (s != CP_OK) return s;
  if (pgrad && !aligned16(pgrad)) return fail(CP_ERR_ALIGNMENT, "prefix_grad_per_rank alignment");
  if (out_lo && dt != CP_BF16) return fail(CP_ERR_DTYPE, "out_lo is for bf16 outputs only");
  if (out_lo && !aligned16(out_lo)) return fail(CP_ERR_ALIGNMENT, "out_lo alignment");
  std::shared_ptr<PlanSet> ps;
  s = get_plans(cu, n_seqs, N, P, T, H, d, &ps);
  if (s != CP_OK) return s;
  if (T == 0) return CP_OK;
  const bool bf16 = dt == CP_BF16;
  const bool tc = bf16;   // bf16: tensor cores (head_dim 64 and 128); fp32: CUDA cores
  if (tc && (s = check_device_for_bf16()) != CP_OK) return s;
  // above softmax scale 0.25: S^T, dQ and dK on f16 operands (scaled copies of Q, K)
  const bool f16 = tc && uses_f16_operands(scale);
  const BwdWs L = bwd_layout(*ps, H, Hkv, d, !tc, !tc && pgrad == nullptr, f16);
  if (!ws || ws_bytes < L.total)
    return fail(CP_ERR_WORKSPACE, "workspace smaller than cp_attn_bwd_workspace_size()");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(CP_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const Problem& pb = ps->pb;
  const int64_t pre_rows = (int64_t)n_seqs * N;
  float* slots = pgrad ? pgrad : reinterpret_cast<float*>(w + L.slots);
  float* pre_k = slots;
  float* pre_v = slots + (size_t)(P + 1) * pre_rows * Hkv * d;
  float* Dd = reinterpret_cast<float*>(w + L.D);
  float* lse2 = reinterpret_cast<float*>(w + L.lse2);
  CP_CUDA(cudaMemsetAsync(w + L.status, 0, kStatusBytes, st), "clear status");
  // tensor cores: one launch over the all-steps plan; CUDA cores: per step.
  // Without per-rank prefix gradients the tensor-core plan sums each prefix
  // key tile's rank terms on chip (one item, natural rows): no slots, no
  // separate sum.
  const bool slots_used = !tc || pgrad != nullptr;
  const FusedBwdPlan& fb = pgrad ? ps->bwd_fused : ps->bwd_fused_merged;
  const std::vector<BwdItem>& bitems = tc ? fb.items : ps->bwd.items;
  CP_CUDA(stager().upload(w + L.items, bitems.data(), bitems.size() * sizeof(BwdItem), st),
          "upload work list");
  if (tc)
    CP_CUDA(stager().upload(w + L.runs, fb.runs.data(), fb.runs.size() * sizeof(Seg), st),
            "upload run list");
  CP_CUDA(stager().upload(w + L.cu, pb.cu.data(), pb.cu.size() * 4, st), "upload cu_seqlens");
  const int64_t pitch = ld_pitch(T);
  OpScales* sc = reinterpret_cast<OpScales*>(w + L.scales);
  void* q16 = w + L.q16;
  void* k16 = w + L.k16;
  {
    ProfScope ps_(3, st, f16 ? 3 : 1);
    CP_CUDA(launch_bwd_preprocess(out, out_lo, dout, bf16, lse, T, H, d, Dd, lse2, pitch, st),
            "bwd preprocess");
    if (f16) {   // max |Q|, |K|, |V|, |dO|; then Q, K * 2^-e in f16 and the factors
      const void* srcs[4] = {q, k, v, dout};
      void* dsts[2] = {q16, k16};
      const int64_t n[4] = {(int64_t)T * H * d, (int64_t)T * Hkv * d, (int64_t)T * Hkv * d,
                            (int64_t)T * H * d};
      CP_CUDA(cudaMemsetAsync(sc, 0, sizeof(OpScales), st), "clear operand scales");
      CP_CUDA(launch_absmax_bf16(srcs, n, 4, sc, st), "max |Q|, |K|, |V|, |dO|");
      CP_CUDA(launch_to_f16_scaled(srcs, dsts, n, 2, sc, true, d, st), "f16 copies of Q, K");
    }
  }
  const BwdItem* items = reinterpret_cast<const BwdItem*>(w + L.items);
  if (tc) {
    CP_CUDA(cudaMemsetAsync(dq, 0, (size_t)T * H * d * sizeof(float), st), "clear dq");
    // With grouped KV heads one CTA walks all G query heads of its KV head.
    // When that leaves too few CTAs to fill the GPU (under ~4 per SM), the
    // group is shared by kv_split CTAs whose partial dK / dV are reduce-added
    // into zeroed memory.
    const int G = H / Hkv;
    int kv_split = 1;
    {
      int dev = 0, sms = 0;
      CP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
      CP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
      const double per_launch = (double)bitems.size() * Hkv;
      while (G % (2 * kv_split) == 0 && per_launch * kv_split < 4.0 * sms) kv_split *= 2;
    }
    if (kv_split > 1) {
      CP_CUDA(cudaMemsetAsync(dk, 0, (size_t)T * Hkv * d * sizeof(float), st), "clear dk");
      CP_CUDA(cudaMemsetAsync(dv, 0, (size_t)T * Hkv * d * sizeof(float), st), "clear dv");
      if (N > 0 && slots_used)
        CP_CUDA(cudaMemsetAsync(slots, 0, 2 * (size_t)(P + 1) * pre_rows * Hkv * d * sizeof(float),
                                st),
                "clear prefix slots");
    }
    TcBwdArgs a;
    const char* terr = nullptr;
    constexpr int tq = 128;   // query rows per tile
    bool ok = make_tmap_thd(&a.tm_q, f16 ? q16 : q, T, H, d, tq, &terr, f16) &&
              make_tmap_thd(&a.tm_k, f16 ? k16 : k, T, Hkv, d, kBwdTileK, &terr, f16) &&
              make_tmap_thd(&a.tm_v, v, T, Hkv, d, kBwdTileK, &terr) &&
              make_tmap_thd(&a.tm_do, dout, T, H, d, tq, &terr) &&
              make_tmap_ld(&a.tm_ld, lse2, pitch, H, tq + 4, &terr) &&
              make_tmap_f32_sw128(&a.tm_dq, dq, T, H, d, 32, &terr);
    if (!ok) return fail(CP_ERR_CUDA, std::string("tensor map: ") + (terr ? terr : "?"));
    a.H = H; a.Hkv = Hkv; a.kv_split = kv_split; a.d = d; a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.T = T;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.pre_k = pre_k; a.pre_v = pre_v; a.pre_rows = pre_rows;
    a.n_slots = P + 1;
    a.status = reinterpret_cast<int32_t*>(w + L.status);
    a.wait_limit = wait_limit();
    a.runs = reinterpret_cast<const Seg*>(w + L.runs);
    a.f16 = f16 ? 1 : 0;
    a.op_scales = f16 ? sc : nullptr;
    // every ring step in one launch: dK / dV summed on chip and written once
    a.items = items;
    a.n_items = (int)bitems.size();
    ProfScope ps_(4, st, 1);
    CP_CUDA(launch_tc_bwd_q128(a, st), "tensor-core backward (all ring steps)");
  } else {
    CP_CUDA(stager().upload(w + L.qitems, ps->fwd_nat.items.data(),
                            ps->fwd_nat.items.size() * sizeof(FwdItem), st),
            "upload dq work list");
    const FwdItem* qitems = reinterpret_cast<const FwdItem*>(w + L.qitems);
    SimtBwdArgs a;
    a.q = q; a.k = k; a.v = v; a.dout = dout; a.D = Dd; a.lse2 = lse2; a.pitch = pitch;
    a.H = H; a.Hkv = Hkv; a.d = d; a.scale = scale; a.T = T;
    a.dq = dq; a.dk = dk; a.dv = dv; a.pre_k = pre_k; a.pre_v = pre_v; a.pre_rows = pre_rows;
    for (int step = 0; step < P; ++step) {
      a.q_items = qitems + ps->fwd_nat.step_begin[step];
      a.n_q_items = ps->fwd_nat.step_begin[step + 1] - ps->fwd_nat.step_begin[step];
      a.k_items = items + ps->bwd.step_begin[step];
      a.n_k_items = ps->bwd.step_begin[step + 1] - ps->bwd.step_begin[step];
      ProfScope ps_(7, st);
      CP_CUDA(launch_simt_bwd_dq(a, st), "backward dq step");
      CP_CUDA(launch_simt_bwd_dkdv(a, st), "backward dk/dv step");
    }
  }
  if (N > 0 && slots_used) {
    // the AllReduce of the replicated prefix gradient: fixed-order sum of slots
    ProfScope ps_(5, st);
    CP_CUDA(launch_prefix_reduce(pre_k, pre_v, P + 1, reinterpret_cast<const int32_t*>(w + L.cu),
                                 n_seqs, N, Hkv, d, dk, dv, st),
            "prefix gradient sum");
  }
  return CP_OK;
}

cp_status_t cp_workspace_status(const void* ws, void* stream) {
  CP_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream sync");
  DevStatus h{};
  if (ws) {
    CP_CUDA(cudaMemcpy(&h, ws, sizeof(int32_t) * 2, cudaMemcpyDeviceToHost), "read status");
  } else {  // the fixed scratch of cp_attn_fwd_noalloc on the current device
    CP_CUDA(noalloc_read_status(&h.timeout), "read the fixed scratch's status");
  }
  if (h.timeout == kStatusBounds) {
    char buf[96];
    snprintf(buf, sizeof buf, "an index outside its tensor was skipped (site %d)", h.where);
    return fail(CP_ERR_BOUNDS, buf);
  }
  if (h.timeout) {
    char buf[96];
    snprintf(buf, sizeof buf, "a device wait gave up (site %d)", h.where);
    return fail(CP_ERR_TIMEOUT, buf);
  }
  return CP_OK;
}

void cp_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
  g_prof_on.store(true);
}

cp_status_t cp_profile_end(double* ms, int64_t* launches) {
  g_prof_on.store(false);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int k = 0; k < kProfKinds; ++k) {
    if (ms) ms[k] = 0.0;
    if (launches) launches[k] = 0;
  }
  cp_status_t st = CP_OK;
  for (auto& r : g_prof) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
    if (e != cudaSuccess) st = cuda_fail(e, "profile events");
    if (r.kind >= 0 && r.kind < kProfKinds) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += r.count;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
  return st;
}

cp_status_t cp_plan_pairs(const int32_t* cu, int n_seqs, int N, int P, int64_t* fwd_pairs,
                          int64_t* bwd_pairs, int64_t* fwd_items, int64_t* bwd_items) {
  if (!cu || n_seqs < 1 || P < 1 || N < 0) return fail(CP_ERR_INVALID_ARG, "bad arguments");
  Problem pb;
  std::string err = make_problem(cu, n_seqs, N, P, -1, &pb);
  if (!err.empty()) return fail(CP_ERR_SHAPE, err);
  // forward: the 256-row items of the tensor-core kernel, checked against the
  // 128-row items of the CUDA-core kernel (both must cover the same pairs),
  // and the all-steps items against the sum over the ring steps
  FwdPlan f, f1;
  FusedFwdPlan fu;
  BwdPlan b;
  FusedBwdPlan bu, bm;
  plan_forward(pb, true, &f, kFwdPairQ);
  plan_forward(pb, true, &f1, kFwdTileQ);
  plan_forward_fused(f, P, &fu);
  plan_backward(pb, &b);
  plan_backward_fused(b, P, 128, false, &bu);
  plan_backward_fused(b, P, 128, true, &bm);
  auto run_pairs = [](const Seg& sg, int q_len) {
    int64_t n = 0;
    for (int t = 0; t < q_len; ++t)
      n += sg.causal ? std::min<int64_t>(sg.len, std::max<int64_t>(0, t + sg.delta + 1)) : sg.len;
    return n;
  };
  auto fwd_step_pairs = [&](const FwdPlan& fp_, int s) {
    int64_t n = 0;
    for (int x = fp_.step_begin[s]; x < fp_.step_begin[s + 1]; ++x) {
      const FwdItem& it = fp_.items[x];
      for (int g = 0; g < it.nseg; ++g) n += run_pairs(it.seg[g], it.q_len);
    }
    return n;
  };
  auto key_pairs = [](const BwdItem& it, const Seg* segs) {
    int64_t n = 0;
    for (int u = 0; u < it.k_len; ++u)
      for (int g = 0; g < it.nseg; ++g) {
        const Seg& sg = segs[g];
        n += sg.causal ? std::max<int64_t>(0, sg.len - std::max<int64_t>(0, u - sg.delta)) : sg.len;
      }
    return n;
  };
  int64_t bwd_fused_pairs = 0, bwd_merged_pairs = 0, bwd_step_sum = 0;
  for (const FusedBwdPlan* plan : {&bu, &bm}) {
    std::map<std::tuple<int32_t, int32_t, int32_t>, int> seen;
    int64_t& sum = plan == &bu ? bwd_fused_pairs : bwd_merged_pairs;
    for (const BwdItem& it : plan->items) {
      if (it.flags != F_FIRST || it.run0 < 0 || it.run0 + it.nseg > (int64_t)plan->runs.size() ||
          seen[std::make_tuple(it.dk_mode, it.k_row0, it.slot)]++ > 0 ||
          (plan == &bm && it.dk_mode != DK_TEXT))
        return fail(CP_ERR_UNSUPPORTED, "all-steps backward item with a bad run range");
      sum += key_pairs(it, plan->runs.data() + it.run0);
    }
  }
  int64_t fused_pairs = 0, step_sum = 0;
  for (const FwdItem& it : fu.items) {
    if (it.flags != (F_FIRST | F_FINAL) || it.run_row0 < 0 ||
        it.run_row0 + it.nseg > (int64_t)fu.runs.size())
      return fail(CP_ERR_UNSUPPORTED, "all-steps forward item with a bad run range");
    for (int g = 0; g < it.nseg; ++g) fused_pairs += run_pairs(fu.runs[it.run_row0 + g], it.q_len);
  }
  for (int s = 0; s < P; ++s) {
    int64_t fp = fwd_step_pairs(f, s), bp = 0;
    if (fp != fwd_step_pairs(f1, s))
      return fail(CP_ERR_UNSUPPORTED, "forward work lists of 128- and 256-row items disagree");
    for (int x = b.step_begin[s]; x < b.step_begin[s + 1]; ++x)
      bp += key_pairs(b.items[x], b.items[x].seg);
    step_sum += fp;
    bwd_step_sum += bp;
    if (fwd_pairs) fwd_pairs[s] = fp;
    if (bwd_pairs) bwd_pairs[s] = bp;
    if (fwd_items) fwd_items[s] = f.step_begin[s + 1] - f.step_begin[s];
    if (bwd_items) bwd_items[s] = b.step_begin[s + 1] - b.step_begin[s];
  }
  if (fused_pairs != step_sum)
    return fail(CP_ERR_UNSUPPORTED, "all-steps forward items disagree with the ring steps");
  if (bwd_fused_pairs != bwd_step_sum || bwd_merged_pairs != bwd_step_sum)
    return fail(CP_ERR_UNSUPPORTED, "all-steps backward items disagree with the ring steps");
  return CP_OK;
}

cp_status_t cp_plan_unit_lists(const int32_t* cu, int n_seqs, int N, int P, int H, int grid,
                               int64_t* n_items, int32_t* tiles, int32_t* units,
                               int32_t* cta_off) {
  if (!cu || n_seqs < 1 || P < 1 || N < 0 || H < 1 || grid < 1)
    return fail(CP_ERR_INVALID_ARG, "bad arguments");
  Problem pb;
  std::string err = make_problem(cu, n_seqs, N, P, -1, &pb);
  if (!err.empty()) return fail(CP_ERR_SHAPE, err);
  FwdPlan f;
  FusedFwdPlan fu;
  plan_forward(pb, true, &f, kFwdPairQ);
  plan_forward_fused(f, P, &fu);
  if ((int64_t)fu.items.size() * H > 0x7fffffffLL)
    return fail(CP_ERR_INVALID_ARG, "too many units");
  if (n_items) *n_items = (int64_t)fu.items.size();
  if (tiles)
    for (size_t x = 0; x < fu.items.size(); ++x) tiles[x] = fu.items[x].n_tiles;
  if (units || cta_off) {
    std::vector<int32_t> u, off;
    plan_unit_lists(fu.items, H, grid, &u, &off);
    if (units) std::copy(u.begin(), u.end(), units);
    if (cta_off) std::copy(off.begin(), off.end(), cta_off);
  }
  return CP_OK;
}

}  // extern "C"
