// Work lists of the chunked tensor-core path and how they are dealt to the
// persistent CTAs or CTA pairs (host code, included by dmuon_api.cu).  What
// is here decides which tiles run together, and with it the L2 reuse and the
// DRAM traffic of the product kernels.
#pragma once

#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/dmuon.h"
#include "common.cuh"
#include "gram.cuh"

namespace dmuon {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }

struct Layout {
  std::vector<MatDesc> mats;       // device pointers filled in once allocated
  std::vector<int64_t> xoff, aoff, boff;  // workspace byte offsets
  std::vector<int64_t> goff;       // Gram-space buffers: kGramBufs per matrix (gram plans)
  std::vector<int64_t> tile_prefix;
  size_t ws_bytes = 0;             // big fp16 workspace
  std::vector<int4> items[3];
  std::vector<int> starts[3];      // per processor: first item of its run (procs + 1 entries)
  int procs[3] = {0, 0, 0};        // persistent CTAs (or CTA pairs) to launch per phase
};

// Cost of one work item for the dealing below, in K-blocks: its main loop,
// but at least the time of a 256 x 256 epilogue (reading, writing and
// mirroring a tile takes about as long as 30-45 K-blocks of products, so a
// short-K tile is epilogue-bound), plus a little for the tile's start.
constexpr int64_t kItemFloor = 32;
constexpr int64_t kItemOverhead = 2;
inline int64_t item_cost(const int4& it) { return std::max<int64_t>(it.w, kItemFloor) + kItemOverhead; }

// Deals a work list over `procs` persistent processors, longest item first,
// each item to the processor with the least work so far (ties: the lowest
// index), and regroups the list so that processor c's items, in the order it
// got them, are [starts[c], starts[c+1]).  A run of equal items falls
// round-robin, as a plain strided dealing would; mixed lengths (gate/up/down
// Grams of K = 14336 beside q/k/v/o ones of K = 4096) no longer leave
// the processors that drew one long item more than the others idle at the end.
// Unbalanced (`balanced` false): the sorted list as is, item w to processor
// w mod procs, and `starts` left empty (the kernels then stride).
inline void deal_items(std::vector<int4>& items, int procs, bool balanced, std::vector<int>& starts, int& used) {
  const int n = (int)items.size();
  used = std::max(0, std::min(procs, n));
  std::stable_sort(items.begin(), items.end(), [](const int4& x, const int4& y) { return x.w > y.w; });
  starts.clear();
  if (used == 0 || !balanced) return;
  starts.assign(used + 1, 0);
  using Load = std::pair<int64_t, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> q;
  for (int c = 0; c < used; ++c) q.push({0, c});
  std::vector<std::vector<int4>> per(used);
  for (const int4& it : items) {
    const Load l = q.top();
    q.pop();
    per[l.second].push_back(it);
    q.push({l.first + item_cost(it), l.second});
  }
  int k = 0;
  for (int c = 0; c < used; ++c) {
    starts[c] = k;
    for (const int4& it : per[c]) items[k++] = it;
  }
  starts[used] = k;
}

// Workspace of a chunk.  Direct plans: X[0], X[1] (m x n fp16), A, B
// (m x m fp16) per matrix.  Gram plans: X[0], X[1] and the kGramBufs m x m
// fp16 buffers of the Gram-space window (R[2], Z[2], W, Q[2], the window's
// last Q).
// bn (single CTAs only): 256 for 128 x 256 tiles, 128 for 128 x 128 tiles.
inline void make_layout(const dmuon_shape_t* shapes, int n, Layout& L, bool pair, int procs, bool balanced,
                 bool gram = false, int bn = kBN) {
  L.mats.assign(n, MatDesc{});
  L.xoff.resize(n); L.aoff.resize(n); L.boff.resize(n);
  L.goff.assign(gram ? (size_t)n * kGramBufs : 0, -1);
  L.tile_prefix.assign(n + 1, 0);
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += (size_t)rup((int64_t)bytes, 256); return (int64_t)o; };
  for (int i = 0; i < n; ++i) {
    MatDesc& d = L.mats[i];
    d.rows = shapes[i].rows;
    d.cols = shapes[i].cols;
    d.transposed = d.rows > d.cols ? 1 : 0;
    d.m = std::min(d.rows, d.cols);
    d.n = std::max(d.rows, d.cols);
    d.ldx = rup(d.n, 8);
    d.lda = rup(d.m, 8);
    d.kappa = scale_kappa(d.m);
    d.beta = scale_beta(d.n);
    L.xoff[i] = take((size_t)(2 * d.m * d.ldx * 2));  // X[0] and X[1] back to back
    if (gram) {
      for (int b = 0; b < kGramBufs; ++b) L.goff[(size_t)i * kGramBufs + b] = take((size_t)(d.m * d.lda * 2));
      L.aoff[i] = L.boff[i] = L.goff[(size_t)i * kGramBufs + kGbQb];
    } else {
      L.aoff[i] = take((size_t)(d.m * d.lda * 2));
      L.boff[i] = take((size_t)(d.m * d.lda * 2));
    }
    d.tiles_c = (int32_t)cdiv(d.cols, kMomTile);
    d.tile0 = L.tile_prefix[i];
    L.tile_prefix[i + 1] = L.tile_prefix[i] + cdiv(d.rows, kMomTile) * d.tiles_c;
  }
  L.ws_bytes = off;
  // Work lists.  Symmetric phases: 256x256 super-tiles (I <= J); Apply: the
  // m x n output.  CTA pairs take a whole 256x256 tile per item; single CTAs
  // take one 128-row half of it, or with 128-column tiles a 128 x 128 block.
  for (int p = 0; p < 3; ++p) L.items[p].clear();
  for (int i = 0; i < n; ++i) {
    MatDesc& d = L.mats[i];
    const size_t sym0 = L.items[kPhaseGram].size(), app0 = L.items[kPhaseApply].size();
    const int64_t T = cdiv(d.m, 256);
    const int kg = (int)cdiv(d.n, kBK), km = (int)cdiv(d.m, kBK);
    if (pair) {
      for (int64_t I = 0; I < T; ++I)
        for (int64_t J = I; J < T; ++J) {
          L.items[kPhaseGram].push_back(make_int4(i, (int)I, (int)J, kg));
          L.items[kPhaseGram2].push_back(make_int4(i, (int)I, (int)J, km));
        }
      for (int64_t tj = 0; tj < cdiv(d.n, kBN); ++tj)
        for (int64_t I = 0; I < T; ++I)
          L.items[kPhaseApply].push_back(make_int4(i, (int)I, (int)tj, km));
      d.sym_items = (int32_t)(L.items[kPhaseGram].size() - sym0);
      d.apply_items = (int32_t)(L.items[kPhaseApply].size() - app0);
      continue;
    }
    if (bn == kBM) {
      // 128 x 128 tiles: blocks (I, J) with I <= J; those above the diagonal
      // also store their transpose.
      const int64_t T1 = cdiv(d.m, kBM);
      for (int64_t I = 0; I < T1; ++I)
        for (int64_t J = I; J < T1; ++J) {
          L.items[kPhaseGram].push_back(make_int4(i, (int)I, (int)J, kg));
          L.items[kPhaseGram2].push_back(make_int4(i, (int)I, (int)J, km));
        }
    } else {
      for (int64_t I = 0; I < T; ++I)
        for (int64_t J = I; J < T; ++J)
          for (int h = 0; h < 2; ++h) {
            const int64_t ti = 2 * I + h;
            if (ti * kBM >= d.m) continue;
            L.items[kPhaseGram].push_back(make_int4(i, (int)ti, (int)J, kg));
            L.items[kPhaseGram2].push_back(make_int4(i, (int)ti, (int)J, km));
          }
    }
    // Column-panel-major: CTAs running together share column panels of X
    // (each read from DRAM once) while B (m x m) stays resident in L2.
    for (int64_t tj = 0; tj < cdiv(d.n, bn); ++tj)
      for (int64_t ti = 0; ti < cdiv(d.m, kBM); ++ti)
        L.items[kPhaseApply].push_back(make_int4(i, (int)ti, (int)tj, km));
    d.sym_items = (int32_t)(L.items[kPhaseGram].size() - sym0);
    d.apply_items = (int32_t)(L.items[kPhaseApply].size() - app0);
  }
  for (int p = 0; p < 3; ++p) deal_items(L.items[p], procs, balanced, L.starts[p], L.procs[p]);
}

}  // namespace dmuon
