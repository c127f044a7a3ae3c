// Host planner: zigzag tables and the per-step work lists.
#include "plan.h"

#include <algorithm>
#include <cstdio>
#include <map>
#include <queue>
#include <tuple>

namespace cpattn {

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rank that holds chunk `slot` (0: chunk r, 1: chunk 2P-1-r) of rank r.
inline int chunk_id(int P, int r, int slot) { return slot == 0 ? r : 2 * P - 1 - r; }

struct Geo {
  const Problem& pb;
  bool text_perm;
  int64_t text0(int i) const { return pb.cu[i] + pb.N; }  // natural row of first text token
  // Row of chunk (rank r, slot) of sample i in the text source tensor.
  int64_t chunk_row(int i, int r, int slot) const {
    if (text_perm) return (int64_t)r * pb.R + pb.off[i] + (int64_t)slot * pb.c[i];
    return text0(i) + (int64_t)chunk_id(pb.P, r, slot) * pb.c[i];
  }
  int32_t text_src() const { return text_perm ? SRC_TEXT : SRC_NAT; }
};

Seg make_seg(int64_t row0, int64_t len, int32_t src, bool causal, int64_t delta) {
  Seg s{};
  s.row0 = (int32_t)row0;
  s.len = (int32_t)len;
  s.src = src;
  s.causal = causal ? 1 : 0;
  s.delta = (int32_t)delta;
  return s;
}

// Visible keys of a run for a query tile of q_len rows (causal: u <= t + delta).
int64_t fwd_visible(const Seg& s, int q_len) {
  if (!s.causal) return s.len;
  return std::max<int64_t>(0, std::min<int64_t>(s.len, (int64_t)q_len + s.delta));
}

// Query rows of a run that see at least one key of a key tile (causal: t >= -delta).
int64_t bwd_visible(const Seg& s) {
  if (!s.causal) return s.len;
  return std::max<int64_t>(0, s.len - std::max<int64_t>(0, -(int64_t)s.delta));
}

}  // namespace

std::string make_problem(const int32_t* cu, int n_seqs, int prefix_len, int P, int T,
                         Problem* out) {
  char buf[256];
  if (!cu) return "cu_seqlens is NULL";
  if (n_seqs < 1) return "n_seqs must be >= 1";
  if (P < 1 || P > 64) return "P must be in [1, 64]";
  if (prefix_len < 0) return "prefix_len must be >= 0";
  if (cu[0] != 0) return "cu_seqlens[0] must be 0";
  Problem pb;
  pb.T = cu[n_seqs];  // plans are cached per cu_seqlens: never the caller's T
  pb.P = P;
  pb.N = prefix_len;
  pb.n_seqs = n_seqs;
  pb.cu.assign(cu, cu + n_seqs + 1);
  int64_t off = 0;
  for (int i = 0; i < n_seqs; ++i) {
    int64_t L = (int64_t)cu[i + 1] - cu[i] - prefix_len;
    if (L < 0) {
      snprintf(buf, sizeof buf, "sample %d is shorter than the prefix (%d tokens)", i,
               prefix_len);
      return buf;
    }
    if (L % (2 * P) != 0) {
      snprintf(buf, sizeof buf, "text length %lld of sample %d is not divisible by 2P=%d",
               (long long)L, i, 2 * P);
      return buf;
    }
    pb.c.push_back((int32_t)(L / (2 * P)));
    pb.off.push_back((int32_t)off);
    off += 2 * (L / (2 * P));
  }
  if (T >= 0 && cu[n_seqs] != T) {
    snprintf(buf, sizeof buf, "cu_seqlens[n_seqs]=%d differs from T=%d", cu[n_seqs], T);
    return buf;
  }
  pb.R = off;
  pb.text_rows = off * P;
  *out = std::move(pb);
  return "";
}

void zigzag_tables(const Problem& pb, int32_t* fwd_idx, int32_t* inv_idx) {
  const int P = pb.P;
  int64_t k = 0;
  // text ordinal of the first text token of each sample
  std::vector<int64_t> ord0(pb.n_seqs, 0);
  for (int i = 1; i < pb.n_seqs; ++i) ord0[i] = ord0[i - 1] + 2LL * P * pb.c[i - 1];
  for (int r = 0; r < P; ++r) {
    for (int i = 0; i < pb.n_seqs; ++i) {
      const int64_t c = pb.c[i];
      const int64_t t0 = (int64_t)pb.cu[i] + pb.N;
      for (int slot = 0; slot < 2; ++slot) {
        const int64_t ch = chunk_id(P, r, slot);
        for (int64_t t = 0; t < c; ++t, ++k) {
          if (fwd_idx) fwd_idx[k] = (int32_t)(t0 + ch * c + t);
          if (inv_idx) inv_idx[ord0[i] + ch * c + t] = (int32_t)k;
        }
      }
    }
  }
}

void plan_forward(const Problem& pb, bool text_perm, FwdPlan* plan, int tile_q) {
  const int P = pb.P;
  Geo g{pb, text_perm};
  plan->items.clear();
  plan->step_begin.assign(1, 0);
  for (int s = 0; s < P; ++s) {
    std::vector<FwdItem> step;
    if (s == 0) {
      // prefix queries: causal self-attention of the prefix, computed once
      for (int i = 0; i < pb.n_seqs && pb.N > 0; ++i) {
        for (int64_t t0 = 0; t0 < pb.N; t0 += tile_q) {
          FwdItem it{};
          it.q_row0 = (int32_t)(pb.cu[i] + t0);
          it.q_len = (int32_t)std::min<int64_t>(tile_q, pb.N - t0);
          it.q_src = SRC_NAT;
          it.seg[0] = make_seg(pb.cu[i], pb.N, SRC_NAT, true, t0);
          it.nseg = 1;
          it.run_row0 = -1;
          it.out_row0 = it.q_row0;
          it.flags = F_FIRST | F_FINAL;
          it.n_tiles = (int32_t)cdiv(fwd_visible(it.seg[0], it.q_len), kFwdTileK);
          step.push_back(it);
        }
      }
    }
    for (int i = 0; i < pb.n_seqs; ++i) {
      const int64_t c = pb.c[i];
      if (c == 0) continue;
      for (int r = 0; r < P; ++r) {
        const int j = ((r - s) % P + P) % P;
        for (int w = 0; w < 2; ++w) {
          const int cq = chunk_id(P, r, w);
          // last ring step at which this query chunk meets a visible key chunk
          int last = 0;
          for (int s2 = 1; s2 < P; ++s2) {
            const int j2 = ((r - s2) % P + P) % P;
            if (chunk_id(P, j2, 0) < cq || chunk_id(P, j2, 1) < cq) last = s2;
          }
          for (int64_t t0 = 0; t0 < c; t0 += tile_q) {
            FwdItem it{};
            it.q_len = (int32_t)std::min<int64_t>(tile_q, c - t0);
            it.q_row0 = (int32_t)(g.chunk_row(i, r, w) + t0);
            it.q_src = g.text_src();
            int n = 0;
            if (s == 0) {
              if (pb.N > 0) it.seg[n++] = make_seg(pb.cu[i], pb.N, SRC_NAT, false, 0);
              for (int w2 = 0; w2 < 2; ++w2) {
                const int ck = chunk_id(P, r, w2);
                if (ck < cq) it.seg[n++] = make_seg(g.chunk_row(i, r, w2), c, g.text_src(), false, 0);
                else if (ck == cq) it.seg[n++] = make_seg(g.chunk_row(i, r, w2), c, g.text_src(), true, t0);
              }
            } else {
              for (int w2 = 0; w2 < 2; ++w2) {
                const int ck = chunk_id(P, j, w2);
                if (ck < cq) it.seg[n++] = make_seg(g.chunk_row(i, j, w2), c, g.text_src(), false, 0);
              }
            }
            if (n == 0) continue;
            it.nseg = n;
            it.run_row0 = (int32_t)((int64_t)r * pb.R + pb.off[i] + w * c + t0);
            it.out_row0 = (int32_t)(g.text0(i) + (int64_t)cq * c + t0);
            it.flags = (s == 0 ? F_FIRST : 0) | (s == last ? F_FINAL : 0);
            int64_t tiles = 0;
            for (int q = 0; q < n; ++q) tiles += cdiv(fwd_visible(it.seg[q], it.q_len), kFwdTileK);
            it.n_tiles = (int32_t)tiles;
            step.push_back(it);
          }
        }
      }
    }
    std::stable_sort(step.begin(), step.end(),
                     [](const FwdItem& a, const FwdItem& b) { return a.n_tiles > b.n_tiles; });
    plan->items.insert(plan->items.end(), step.begin(), step.end());
    plan->step_begin.push_back((int32_t)plan->items.size());
  }
}

void plan_forward_fused(const FwdPlan& per_step, int P, FusedFwdPlan* out) {
  // group the per-step items by query tile, keeping ring-step order
  struct Acc {
    FwdItem head;
    std::vector<Seg> segs;
  };
  std::vector<Acc> acc;
  std::map<std::pair<int32_t, int32_t>, size_t> where;  // (q_src, q_row0) -> acc index
  for (int s = 0; s < P; ++s) {
    for (int x = per_step.step_begin[s]; x < per_step.step_begin[s + 1]; ++x) {
      const FwdItem& it = per_step.items[x];
      const auto key = std::make_pair(it.q_src, it.q_row0);
      auto f = where.find(key);
      if (f == where.end()) {
        f = where.emplace(key, acc.size()).first;
        acc.push_back({it, {}});
      }
      for (int g = 0; g < it.nseg; ++g) acc[f->second].segs.push_back(it.seg[g]);
    }
  }
  out->items.clear();
  out->runs.clear();
  for (Acc& a : acc) {
    FwdItem it = a.head;
    it.nseg = (int32_t)a.segs.size();
    it.run_row0 = (int32_t)out->runs.size();
    it.flags = F_FIRST | F_FINAL;
    int64_t tiles = 0;
    for (const Seg& sg : a.segs) tiles += cdiv(fwd_visible(sg, it.q_len), kFwdTileK);
    it.n_tiles = (int32_t)tiles;
    out->runs.insert(out->runs.end(), a.segs.begin(), a.segs.end());
    out->items.push_back(it);
  }
  std::stable_sort(out->items.begin(), out->items.end(),
                   [](const FwdItem& a, const FwdItem& b) { return a.n_tiles > b.n_tiles; });
}

void plan_unit_lists(const std::vector<FwdItem>& items, int H, int grid,
                     std::vector<int32_t>* units, std::vector<int32_t>* cta_off) {
  constexpr int64_t kUnitCost = 2;  // Q load and epilogue, in KV-tile equivalents
  const int n = (int)items.size();
  std::vector<std::vector<int32_t>> lists(grid);
  using Load = std::pair<int64_t, int>;  // (work so far, CTA): least work first, then lowest CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> pq;
  for (int b = 0; b < grid; ++b) pq.push({0, b});
  for (int h = 0; h < H; ++h) {
    for (int x = 0; x < n; ++x) {
      Load e = pq.top();
      pq.pop();
      lists[e.second].push_back(x + n * h);
      e.first += items[x].n_tiles + kUnitCost;
      pq.push(e);
    }
  }
  units->clear();
  cta_off->assign(1, 0);
  for (const auto& l : lists) {
    units->insert(units->end(), l.begin(), l.end());
    cta_off->push_back((int32_t)units->size());
  }
}

void plan_backward(const Problem& pb, BwdPlan* plan) {
  const int P = pb.P;
  Geo g{pb, false};
  plan->items.clear();
  plan->step_begin.assign(1, 0);
  auto finish = [](BwdItem& it) {
    int64_t tiles = 0;
    for (int q = 0; q < it.nseg; ++q) tiles += cdiv(bwd_visible(it.seg[q]), kBwdTileQ);
    it.n_tiles = (int32_t)tiles;
  };
  for (int s = 0; s < P; ++s) {
    std::vector<BwdItem> step;
    for (int i = 0; i < pb.n_seqs; ++i) {
      const int64_t c = pb.c[i];
      if (s == 0 && pb.N > 0) {
        for (int64_t u0 = 0; u0 < pb.N; u0 += kBwdTileK) {
          const int32_t klen = (int32_t)std::min<int64_t>(kBwdTileK, pb.N - u0);
          // per-rank prefix gradient: rank r's text queries see the whole prefix
          for (int r = 0; r <= P; ++r) {
            BwdItem it{};
            it.run0 = -1;
            it.k_row0 = (int32_t)(pb.cu[i] + u0);
            it.k_len = klen;
            it.dk_mode = DK_PREFIX_SLOT;
            it.dk_row0 = (int32_t)((int64_t)i * pb.N + u0);
            it.slot = r;
            it.flags = F_FIRST;
            int n = 0;
            if (r < P) {
              for (int w = 0; w < 2 && c > 0; ++w)
                it.seg[n++] = make_seg(g.chunk_row(i, r, w), c, SRC_NAT, false, 0);
            } else {
              it.seg[n++] = make_seg(pb.cu[i] + u0, pb.N - u0, SRC_NAT, true, 0);
            }
            it.nseg = n;
            finish(it);
            step.push_back(it);
          }
        }
      }
      if (c == 0) continue;
      for (int j = 0; j < P; ++j) {
        const int r = (j + s) % P;  // query rank that meets rank j's KV at step s
        for (int w = 0; w < 2; ++w) {
          const int ck = chunk_id(P, j, w);
          for (int64_t u0 = 0; u0 < c; u0 += kBwdTileK) {
            BwdItem it{};
            it.run0 = -1;
            it.k_row0 = (int32_t)(g.chunk_row(i, j, w) + u0);
            it.k_len = (int32_t)std::min<int64_t>(kBwdTileK, c - u0);
            it.dk_mode = DK_TEXT;
            it.dk_row0 = it.k_row0;
            it.slot = 0;
            it.flags = s == 0 ? F_FIRST : 0;
            int n = 0;
            for (int w2 = 0; w2 < 2; ++w2) {
              const int cq = chunk_id(P, r, w2);
              if (cq > ck) it.seg[n++] = make_seg(g.chunk_row(i, r, w2), c, SRC_NAT, false, 0);
              else if (cq == ck)
                it.seg[n++] = make_seg(g.chunk_row(i, r, w2) + u0, c - u0, SRC_NAT, true, 0);
            }
            if (n == 0) continue;
            it.nseg = n;
            finish(it);
            step.push_back(it);
          }
        }
      }
    }
    std::stable_sort(step.begin(), step.end(),
                     [](const BwdItem& a, const BwdItem& b) { return a.n_tiles > b.n_tiles; });
    plan->items.insert(plan->items.end(), step.begin(), step.end());
    plan->step_begin.push_back((int32_t)plan->items.size());
  }
}

void plan_backward_fused(const BwdPlan& per_step, int P, int tile_q, bool merge_prefix_slots,
                         FusedBwdPlan* out) {
  // group the per-step items by destination (text key tile, or prefix key
  // tile and slot, or prefix key tile alone when the slots merge), keeping
  // ring-step order
  struct Acc {
    BwdItem head;
    std::vector<Seg> segs;
  };
  std::vector<Acc> acc;
  std::map<std::tuple<int32_t, int32_t, int32_t>, size_t> where;  // (dk_mode, k_row0, slot)
  for (int s = 0; s < P; ++s) {
    for (int x = per_step.step_begin[s]; x < per_step.step_begin[s + 1]; ++x) {
      BwdItem it = per_step.items[x];
      if (merge_prefix_slots && it.dk_mode == DK_PREFIX_SLOT) {
        it.dk_mode = DK_TEXT;   // the summed prefix gradient, at its natural rows
        it.dk_row0 = it.k_row0;
        it.slot = 0;
      }
      const auto key = std::make_tuple(it.dk_mode, it.k_row0, it.slot);
      auto f = where.find(key);
      if (f == where.end()) {
        f = where.emplace(key, acc.size()).first;
        acc.push_back({it, {}});
      }
      for (int g = 0; g < it.nseg; ++g) acc[f->second].segs.push_back(it.seg[g]);
    }
  }
  out->items.clear();
  out->runs.clear();
  for (Acc& a : acc) {
    BwdItem it = a.head;
    it.nseg = (int32_t)a.segs.size();
    it.run0 = (int32_t)out->runs.size();
    it.flags = F_FIRST;
    for (int g = 0; g < kBwdMaxSeg; ++g) it.seg[g] = Seg{};
    int64_t tiles = 0;
    for (const Seg& sg : a.segs) tiles += cdiv(bwd_visible(sg), tile_q);
    it.n_tiles = (int32_t)tiles;
    out->runs.insert(out->runs.end(), a.segs.begin(), a.segs.end());
    out->items.push_back(it);
  }
  std::stable_sort(out->items.begin(), out->items.end(),
                   [](const BwdItem& a, const BwdItem& b) { return a.n_tiles > b.n_tiles; });
}

}  // namespace cpattn
