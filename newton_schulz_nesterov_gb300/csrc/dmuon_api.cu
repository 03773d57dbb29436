// Host side of the C ABI declared in include/dmuon.h: argument checks,
// planning (orientation, workspace layout, TMA descriptors, work lists),
// per-call pointer upload and the launch sequence of one step.
//
// Launch sequence of one step (all on the caller's stream, no host sync):
//   ns_small    every small matrix (oriented m <= 128, n <= 512) in one
//               launch, one CTA per matrix running its whole step
//   then, per chunk of the other matrices:
//   mom_norm    M <- mu*M + G, U, X0 = fp16(p U or p U^T), tile sums of
//               (p U)^2 and tile maxima of |U|
//   finalize    s = 1/(||U||_F + eps) per matrix, or a new power of two p
//               for a matrix whose p U missed fp16's comfortable range
//   mom_norm, finalize (redo pass): rewrite X0 of those matrices; both
//               return at once when there are none
//   ns_steps x [ Gram (A = X X^T) -> Gram2 (Z = aI + bA + cAA) -> Apply (X' = Z X) ]
//   the last Apply updates W in place (or writes O for the standalone NS)
// All stored iterates and products are fp16 with power-of-two scales
// (MatDesc); the tensor cores accumulate in fp32.
//
// Plan order: the large matrices (in the caller's order, chunked), then the
// small ones.  Device pointer sets and flags are kept in plan order; the
// caller's order is restored when flags are read.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/dmuon.h"
#include "aux.cuh"
#include "coeffs.cuh"
#include "common.cuh"
#include "gram.cuh"
#include "plan.cuh"
#include "small.cuh"

using namespace dmuon;

namespace {

const char* kVersion = "dmuon-gb300 0.1.0 (sm_103a, tcgen05/TMA)";

// Cached caller pointer sets per plan (see run()).
constexpr int kPtrSlots = 64;

// Shapes the fused small-matrix kernel takes (oriented m <= 128, n <= 512).
inline bool is_small(const dmuon_shape_t& s) {
  return std::min(s.rows, s.cols) <= kSmallMaxM && std::max(s.rows, s.cols) <= kSmallMaxN;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// fp16 row-major rows x cols with leading dimension ld (elements): 64x64
// boxes, 128-byte swizzle, zero fill outside the matrix.
bool encode_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)kBox, (cuuint32_t)kBox};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

struct ProfRec {
  cudaEvent_t a, b;
  int kind;
};

// One chunk of the matrix list: a contiguous run [i0, i0 + n) planned and
// launched as a unit.  All chunks share one workspace and run one after the
// other on the stream.
struct Chunk {
  int i0 = 0, n = 0;
  Layout L;                       // sub-list layout (workspace offsets, work lists)
  MatDesc* d_mats = nullptr;
  CUtensorMap* d_maps = nullptr;
  int64_t* d_prefix = nullptr;
  float* d_partials = nullptr;
  float* d_tmax = nullptr;        // per momentum tile: max |U|
  float* d_svec = nullptr;        // per matrix: s/p
  float* d_bvec = nullptr;        // per matrix: beta', the scale of the iterate after the first product
  float* d_pscale = nullptr;      // per matrix: the prescale p of X[0] (kept across steps)
  int* d_redo = nullptr;          // per matrix: X[0] to be rewritten with a new p
  int* d_counters = nullptr;      // per matrix: finished tiles of a fused launch (zeroed before it)
  int4* d_items[3] = {nullptr, nullptr, nullptr};
  int* d_starts[3] = {nullptr, nullptr, nullptr};
  GramDesc* d_gd = nullptr;       // gram plans: per-matrix Gram-space buffers
  CUtensorMap* d_gmaps = nullptr; // gram plans: kGramBufs maps per matrix
};

struct dmuon_ctx {
  int device = 0;
  int num_sms = 0;
  // plan
  std::vector<dmuon_shape_t> shapes;   // caller order
  std::vector<int> order;              // plan position -> caller index
  int n_large = 0;                     // plan positions [0, n_large) are chunked
  std::vector<SmallDesc> small_descs;  // plan positions [n_large, n)
  SmallDesc* d_small = nullptr;
  bool small_path = true;              // requested
  bool small_ok = false;               // small kernel configured on this device
  bool plan_small = false;             // small kernel used by the current plan
  bool plan_gram = false;              // chunks laid out for the Gram-space backend
  bool gram_ok = false;                // Gram-space kernels configured on this device
  std::vector<Chunk> chunks;
  size_t ws_bytes = 0, small_bytes = 0;
  void* ws = nullptr;
  void* small = nullptr;
  MatPtrs* d_ptrs = nullptr;
  int* d_flags = nullptr;
  int* d_err = nullptr;
  // pointer-set cache: kPtrSlots device slots of n MatPtrs each
  std::vector<MatPtrs> slot_ptrs[kPtrSlots];
  uint64_t slot_use[kPtrSlots] = {};
  bool slot_pending[kPtrSlots] = {};
  cudaEvent_t slot_ev[kPtrSlots] = {};
  uint64_t use_clock = 0;
  MatPtrs* h_stage = nullptr;  // pinned staging, kPtrSlots x n
  cudaStream_t last_stream = nullptr;
  int64_t launches = 0;
  bool profiling = false;
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> ev_pool;
  std::string last_error;
  unsigned long long wait_timeout_ns = 0;  // 0: kernels' default (4 s)
  int max_clusters = 0;                     // resident 2-CTA clusters (0: pairs unavailable)
  int tile_mode = 0;                        // requested: 0 auto, 1 single CTA, 2 CTA pairs, 3 single CTA 128x128
  int64_t chunk_elems = 0;                  // requested chunk size (0: default)
  bool plan_pair = false;                   // tile kind of the current plan
  int plan_bn = kBN;                        // its single-CTA tile width (256, or 128)
  int64_t plan_chunk_elems = 0;             // chunk size of the current plan
  // Overlap of chunk c+1's momentum pass with chunk c's tensor-core phases:
  // a side stream, two alternating chunk workspaces and fork/join events.
  bool overlap = false;                     // requested (off: measured neutral at the power cap)
  bool balanced = true;                     // requested: work items dealt longest-first to the least loaded
  int f16_iters = 3;                        // direct backend: leading iterations with fp16 operands
  int fused = 2;                            // direct backend, one launch per chunk for all products:
                                            // 0 never, 1 always, 2 for chunks of few work items
  bool plan_balanced = true;                // in the current plan
  bool plan_overlap = false;                // in the current plan (needs >= 2 chunks)
  size_t ws_chunk = 0;                      // bytes of one chunk workspace
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_norm[2] = {}, ev_gemm[2] = {};
  // AdamW / clipping: descriptor buffer (device), pinned staging, results
  void* aux_dev = nullptr;
  size_t aux_dev_cap = 0;
  uint8_t* aux_host = nullptr;
  size_t aux_host_cap = 0;
  cudaEvent_t aux_ev = nullptr;
  bool aux_pending = false;
};

namespace {

// Default chunk: up to 2^29 matrix elements (1 GiB per 16-bit iterate buffer).
// Running the 2 + 3*ns_steps launches over a few layers' worth of matrices at
// a time, instead of the whole list, measured ~6 % faster on the Llama-3-8B
// set and bounds the workspace by the largest chunk.
constexpr int64_t kDefaultChunkElems = int64_t(1) << 29;

// Automatic fused launch (dmuon_set_fused_phases mode 2): chunks whose three
// phases hold at most this many work items per persistent processor, where
// launch fills and drains dominate.  Measured on GB300: TinyMLP d=512 (528
// items over 152 CTAs) 0.42 ms per step fused against 0.49 ms per phase; the
// Llama-3-8B set (thousands of items per chunk) 395 ms fused against 330 ms,
// the fused kernel's processors drifting apart across phases and reading 41 %
// more from DRAM.
constexpr int64_t kFuseItemsPerProc = 8;

int cuda_err(cudaError_t e) { return e == cudaSuccess ? DMUON_OK : (e == cudaErrorMemoryAllocation ? DMUON_ERR_OOM : DMUON_ERR_CUDA); }

// Record what failed (readable through dmuon_last_error) and return `code`.
int fail(dmuon_ctx* h, int code, const char* what, cudaError_t e = cudaSuccess) {
  char buf[384];
  if (e != cudaSuccess)
    std::snprintf(buf, sizeof buf, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  else
    std::snprintf(buf, sizeof buf, "%s", what);
  h->last_error = buf;
  return code;
}

void free_plan(dmuon_ctx* h) {
  if (h->ws || h->small) cudaDeviceSynchronize();
  if (h->ws) cudaFree(h->ws);
  if (h->small) cudaFree(h->small);
  h->ws = h->small = nullptr;
  h->shapes.clear();
  h->order.clear();
  h->small_descs.clear();
  h->d_small = nullptr;
  h->n_large = 0;
  h->chunks.clear();
  for (int k = 0; k < kPtrSlots; ++k) {
    if (h->slot_pending[k]) cudaEventSynchronize(h->slot_ev[k]);
    h->slot_pending[k] = false;
    h->slot_ptrs[k].clear();
    h->slot_use[k] = 0;
  }
  if (h->h_stage) cudaFreeHost(h->h_stage);
  h->h_stage = nullptr;
}

// CTA pairs unless single CTAs are requested, pairs are unavailable, or (in
// automatic mode) every short side fits one 128-row tile, where a pair's
// second CTA would only compute padding.
// Dealing quality of phase q of a layout: the busiest processor's summed
// item cost and the mean cost per processor (costs as item_cost).
inline std::pair<double, double> deal_balance(const Layout& L, int q) {
  const int P = L.procs[q], n_it = (int)L.items[q].size();
  if (P <= 0) return {0.0, 0.0};
  const bool strided = L.starts[q].empty();
  double total = 0, top = 0;
  for (int c = 0; c < P; ++c) {
    double run = 0;
    for (int w = strided ? c : L.starts[q][c]; w < (strided ? n_it : L.starts[q][c + 1]); w += strided ? P : 1)
      run += (double)item_cost(L.items[q][w]);
    total += run;
    top = std::max(top, run);
  }
  return {top, total / P};
}

// Tile kind of a plan (max_clusters: resident 2-CTA clusters, 0 if none;
// small_on: the small-matrix kernel takes the small matrices).
bool choose_pairs(int max_clusters, int tile_mode, bool small_on, const dmuon_shape_t* s, int n, bool gram) {
  if (max_clusters <= 0) return false;
  if (gram) return true;  // the Gram-space kernels exist for CTA pairs only
  if (tile_mode == 1 || tile_mode == 3) return false;  // single CTAs, 128 x 256 or 128 x 128
  if (tile_mode == 2) return true;
  // Automatic: pairs once some chunked matrix's short side exceeds one
  // 128-row tile and the chunked matrices give at least one 256 x 256 Gram
  // super-tile per CTA pair.  A list with fewer leaves most pairs idle and
  // its launches are latency-bound; single CTAs (twice the items) finish it
  // sooner (12 TinyMLP d=512 matrices: 0.461 against 0.482 ms per step).
  bool wide = false;
  int64_t items = 0;
  for (int i = 0; i < n; ++i) {
    if (small_on && is_small(s[i])) continue;  // the small-matrix kernel takes it
    const int64_t m = std::min(s[i].rows, s[i].cols), T = cdiv(m, 256);
    wide = wide || m > kBM;
    items += T * (T + 1) / 2;
  }
  return wide && items >= max_clusters;
}

bool use_pairs(const dmuon_ctx* h, const dmuon_shape_t* s, int n, bool gram = false) {
  return choose_pairs(h->max_clusters, h->tile_mode, h->small_path && h->small_ok, s, n, gram);
}

// Single-CTA tile width.  Automatic: 128 x 128 blocks when the 128 x 256
// Gram items of the chunked matrices would leave SMs idle -- such lists are
// latency-bound (short K, exposed epilogues), and blocks of half the width
// double the items and halve each one's epilogue (TinyMLP d=512: 72 items
// of 128 x 256 for 152 SMs).
int choose_bn(int sms, int tile_mode, bool small_on, const dmuon_shape_t* s, int n) {
  if (tile_mode == 3) return kBM;
  if (tile_mode == 1) return kBN;
  int64_t items = 0;
  for (int i = 0; i < n; ++i) {
    if (small_on && is_small(s[i])) continue;
    const int64_t m = std::min(s[i].rows, s[i].cols), T = cdiv(m, 256), halves = cdiv(m, kBM);
    items += T * (T - 1) / 2 * 2 + halves;  // super-tiles above the diagonal: both halves; on it: those inside m
  }
  return items < sms ? kBM : kBN;
}

int use_bn(const dmuon_ctx* h, const dmuon_shape_t* s, int n, bool gram = false) {
  return use_pairs(h, s, n, gram) ? kBN : choose_bn(h->num_sms, h->tile_mode, h->small_path && h->small_ok, s, n);
}

int64_t chunk_limit(const dmuon_ctx* h) { return h->chunk_elems > 0 ? h->chunk_elems : kDefaultChunkElems; }

bool same_shapes(const dmuon_ctx* h, const dmuon_shape_t* s, int n, bool gram = false) {
  if ((int)h->shapes.size() != n || !h->small || h->plan_pair != use_pairs(h, s, n, gram) ||
      h->plan_bn != use_bn(h, s, n, gram) ||
      h->plan_gram != gram ||
      h->plan_small != (h->small_path && h->small_ok) ||
      h->plan_chunk_elems != chunk_limit(h) || h->plan_balanced != h->balanced || h->plan_overlap != (h->overlap && h->chunks.size() > 1))
    return false;
  for (int i = 0; i < n; ++i)
    if (h->shapes[i].rows != s[i].rows || h->shapes[i].cols != s[i].cols) return false;
  return true;
}

// Greedy contiguous chunks of at most `limit` elements (a larger matrix is a
// chunk of its own).
std::vector<std::pair<int, int>> split_chunks(const dmuon_shape_t* shapes, int n, int64_t limit) {
  std::vector<std::pair<int, int>> out;
  int i0 = 0;
  int64_t sum = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t e = shapes[i].rows * shapes[i].cols;
    if (i > i0 && sum + e > limit) {
      out.push_back({i0, i - i0});
      i0 = i;
      sum = 0;
    }
    sum += e;
  }
  if (n > i0) out.push_back({i0, n - i0});
  return out;
}

// Bytes of one chunk's device arrays (descriptors, maps, prefix, tile sums and
// maxima, scale, prescale and redo vectors, work lists).
size_t chunk_small_bytes(const Layout& L, int n) {
  const bool gram = !L.goff.empty();
  return rup(sizeof(MatDesc) * n, 256) + rup(sizeof(CUtensorMap) * kMapsPerMat * n, 256) +
         rup(8 * (n + 1), 256) + 2 * rup(4 * L.tile_prefix[n], 256) + 5 * rup(4 * n, 256) +
         rup(16 * L.items[0].size(), 256) + rup(16 * L.items[1].size(), 256) + rup(16 * L.items[2].size(), 256) +
         rup(4 * (L.items[0].size() + 1), 256) + rup(4 * (L.items[1].size() + 1), 256) +
         rup(4 * (L.items[2].size() + 1), 256) +
         (gram ? rup(sizeof(GramDesc) * n, 256) + rup(sizeof(CUtensorMap) * kGramBufs * n, 256) : 0);
}

// Plan order: positions [0, n_large) hold the matrices run by the chunked
// tensor-core path (caller order), the rest the small ones (caller order).
int plan_order(const dmuon_shape_t* shapes, int n, bool small_path, std::vector<int>& order) {
  order.clear();
  for (int i = 0; i < n; ++i)
    if (!(small_path && is_small(shapes[i]))) order.push_back(i);
  const int n_large = (int)order.size();
  for (int i = 0; i < n; ++i)
    if (small_path && is_small(shapes[i])) order.push_back(i);
  return n_large;
}

// Host-side plan sizes (no device work): workspace of the largest chunk and
// all device arrays, for CTA pairs or single CTAs of tile width bn.
void plan_sizes(const dmuon_shape_t* shapes, int n, bool pair, int64_t limit, bool small_path, size_t* ws,
                size_t* small, bool gram = false, int bn = kBN) {
  std::vector<int> order;
  const int n_large = plan_order(shapes, n, small_path, order);
  std::vector<dmuon_shape_t> ps(n);
  for (int k = 0; k < n; ++k) ps[k] = shapes[order[k]];
  *ws = 256;
  *small = rup(sizeof(MatPtrs) * n * kPtrSlots, 256) + rup(4 * n, 256) + 256 +
           rup(sizeof(SmallDesc) * (n - n_large), 256);
  for (const auto& c : split_chunks(ps.data(), n_large, limit)) {
    Layout L;
    make_layout(ps.data() + c.first, c.second, L, pair, 1, true, gram, bn);  // sizes do not depend on procs
    *ws = std::max(*ws, L.ws_bytes);
    *small += chunk_small_bytes(L, c.second);
  }
}

int build_plan(dmuon_ctx* h, const dmuon_shape_t* shapes, int n, bool gram) {
  if (same_shapes(h, shapes, n, gram)) return DMUON_OK;
  free_plan(h);
  if (!get_encoder()) return fail(h, DMUON_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  if (gram && (h->max_clusters <= 0 || !h->gram_ok))
    return fail(h, DMUON_ERR_UNSUPPORTED, "Gram-space backend needs 2-CTA clusters, unavailable on this device");
  h->plan_gram = gram;
  h->plan_pair = use_pairs(h, shapes, n, gram);
  h->plan_bn = use_bn(h, shapes, n, gram);
  h->plan_chunk_elems = chunk_limit(h);
  h->plan_balanced = h->balanced;
  h->plan_small = h->small_path && h->small_ok;
  h->n_large = plan_order(shapes, n, h->plan_small, h->order);
  std::vector<dmuon_shape_t> ps(n);
  for (int k = 0; k < n; ++k) ps[k] = shapes[h->order[k]];
  const int n_small = n - h->n_large;
  h->small_descs.resize(n_small);
  for (int k = 0; k < n_small; ++k)
    h->small_descs[k] = SmallDesc{ps[h->n_large + k].rows, ps[h->n_large + k].cols, h->n_large + k, 1.f};
  const auto parts = split_chunks(ps.data(), h->n_large, h->plan_chunk_elems);
  h->chunks.resize(parts.size());
  h->ws_bytes = 256;
  h->small_bytes = rup(sizeof(MatPtrs) * n * kPtrSlots, 256) + rup(4 * n, 256) + 256 +
                   rup(sizeof(SmallDesc) * n_small, 256);
  for (size_t c = 0; c < parts.size(); ++c) {
    Chunk& ch = h->chunks[c];
    ch.i0 = parts[c].first;
    ch.n = parts[c].second;
    make_layout(ps.data() + ch.i0, ch.n, ch.L, h->plan_pair, h->plan_pair ? h->max_clusters : h->num_sms,
                h->plan_balanced, gram, h->plan_bn);
    h->ws_bytes = std::max(h->ws_bytes, ch.L.ws_bytes);
    h->small_bytes += chunk_small_bytes(ch.L, ch.n);
  }
  h->ws_chunk = h->ws_bytes;
  h->plan_overlap = h->overlap && h->chunks.size() > 1;
  if (h->plan_overlap) h->ws_bytes = 2 * h->ws_chunk;  // chunks alternate between two
  cudaError_t e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) { h->ws = nullptr; cudaGetLastError(); free_plan(h); return fail(h, DMUON_ERR_OOM, "workspace cudaMalloc", e); }
  e = cudaMalloc(&h->small, h->small_bytes);
  if (e != cudaSuccess) { h->small = nullptr; cudaGetLastError(); free_plan(h); return fail(h, DMUON_ERR_OOM, "descriptor cudaMalloc", e); }
  uint8_t* p = (uint8_t*)h->small;
  auto carve = [&](size_t bytes) { uint8_t* q = p; p += rup((int64_t)bytes, 256); return q; };
  h->d_ptrs = (MatPtrs*)carve(sizeof(MatPtrs) * n * kPtrSlots);
  h->d_flags = (int*)carve(4 * n);
  h->d_err = (int*)carve(256);
  h->d_small = (SmallDesc*)carve(sizeof(SmallDesc) * n_small);
  if (n_small > 0) {
    e = cudaMemcpy(h->d_small, h->small_descs.data(), sizeof(SmallDesc) * n_small, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) { free_plan(h); return fail(h, cuda_err(e), "plan upload", e); }
  }
  for (size_t c = 0; c < h->chunks.size(); ++c) {
    Chunk& ch = h->chunks[c];
    uint8_t* ws = (uint8_t*)h->ws + (h->plan_overlap ? (c & 1) * h->ws_chunk : 0);
    Layout& L = ch.L;
    const int cn = ch.n;
    ch.d_mats = (MatDesc*)carve(sizeof(MatDesc) * cn);
    ch.d_maps = (CUtensorMap*)carve(sizeof(CUtensorMap) * kMapsPerMat * cn);
    ch.d_prefix = (int64_t*)carve(8 * (cn + 1));
    ch.d_partials = (float*)carve(4 * L.tile_prefix[cn]);
    ch.d_tmax = (float*)carve(4 * L.tile_prefix[cn]);
    ch.d_svec = (float*)carve(4 * cn);
    ch.d_bvec = (float*)carve(4 * cn);
    ch.d_pscale = (float*)carve(4 * cn);
    ch.d_redo = (int*)carve(4 * cn);
    ch.d_counters = (int*)carve(4 * cn);
    for (int q = 0; q < 3; ++q) ch.d_items[q] = (int4*)carve(16 * L.items[q].size());
    for (int q = 0; q < 3; ++q) ch.d_starts[q] = (int*)carve(4 * (L.items[q].size() + 1));
    if (gram) {
      ch.d_gd = (GramDesc*)carve(sizeof(GramDesc) * cn);
      ch.d_gmaps = (CUtensorMap*)carve(sizeof(CUtensorMap) * kGramBufs * cn);
    }
    std::vector<CUtensorMap> maps(kMapsPerMat * (size_t)cn);
    std::vector<CUtensorMap> gmaps(gram ? kGramBufs * (size_t)cn : 0);
    std::vector<GramDesc> gds(gram ? cn : 0);
    for (int i = 0; i < cn; ++i) {
      MatDesc& d = L.mats[i];
      d.X[0] = (__half*)(ws + L.xoff[i]);
      d.X[1] = d.X[0] + d.m * d.ldx;
      d.A = (__half*)(ws + L.aoff[i]);
      d.B = (__half*)(ws + L.boff[i]);
      d.scale = 1.f;
      bool ok = encode_map(&maps[kMapsPerMat * i + 0], d.X[0], d.m, d.n, d.ldx) &&
                encode_map(&maps[kMapsPerMat * i + 1], d.X[1], d.m, d.n, d.ldx) &&
                encode_map(&maps[kMapsPerMat * i + 2], d.A, d.m, d.m, d.lda) &&
                encode_map(&maps[kMapsPerMat * i + 3], d.B, d.m, d.m, d.lda);
      if (gram) {
        // Gram plans: A and B above both name the window's last Q, so the
        // direct Apply kernel computes Q X.
        GramDesc& gd = gds[i];
        gd.m = d.m;
        gd.ld = d.lda;
        gd.kappa = d.kappa;
        gd.inv_kappa = 1.f / gd.kappa;
        for (int b = 0; b < kGramBufs && ok; ++b) {
          gd.buf[b] = (uint16_t*)(ws + L.goff[(size_t)i * kGramBufs + b]);
          ok = encode_map(&gmaps[kGramBufs * i + b], gd.buf[b], d.m, d.m, d.lda);
        }
      }
      if (!ok) {
        char what[160];
        std::snprintf(what, sizeof what, "cuTensorMapEncodeTiled failed for matrix %d (%lld x %lld)",
                      h->order[ch.i0 + i],
                      (long long)d.rows, (long long)d.cols);
        free_plan(h);
        return fail(h, DMUON_ERR_CUDA, what);
      }
    }
    e = cudaMemcpy(ch.d_mats, L.mats.data(), sizeof(MatDesc) * cn, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
      const std::vector<float> ones(cn, 1.f);  // first prescale guess; corrected by the first step
      e = cudaMemcpy(ch.d_pscale, ones.data(), 4 * cn, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaMemset(ch.d_redo, 0, 4 * cn);
    if (e == cudaSuccess) e = cudaMemcpy(ch.d_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ch.d_prefix, L.tile_prefix.data(), 8 * (cn + 1), cudaMemcpyHostToDevice);
    if (gram && e == cudaSuccess) e = cudaMemcpy(ch.d_gd, gds.data(), sizeof(GramDesc) * cn, cudaMemcpyHostToDevice);
    if (gram && e == cudaSuccess)
      e = cudaMemcpy(ch.d_gmaps, gmaps.data(), sizeof(CUtensorMap) * gmaps.size(), cudaMemcpyHostToDevice);
    for (int q = 0; q < 3 && e == cudaSuccess; ++q)
      if (!L.items[q].empty()) {
        e = cudaMemcpy(ch.d_items[q], L.items[q].data(), 16 * L.items[q].size(), cudaMemcpyHostToDevice);
        if (e == cudaSuccess && !L.starts[q].empty())
          e = cudaMemcpy(ch.d_starts[q], L.starts[q].data(), 4 * L.starts[q].size(), cudaMemcpyHostToDevice);
      }
    if (e != cudaSuccess) { free_plan(h); return fail(h, cuda_err(e), "plan upload", e); }
  }
  e = cudaMemset(h->d_flags, 0, 4 * n);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, 256);
  if (e != cudaSuccess) { free_plan(h); return fail(h, cuda_err(e), "plan upload", e); }
  if (cudaMallocHost(&h->h_stage, sizeof(MatPtrs) * n * kPtrSlots) != cudaSuccess) {
    h->h_stage = nullptr;
    free_plan(h);
    return fail(h, DMUON_ERR_OOM, "pinned pointer staging");
  }
  h->shapes.assign(shapes, shapes + n);
  return DMUON_OK;
}

// Per-matrix update scale (the pages give none; reading: original Muon
// sqrt(max(1, rows/cols)) by default).
float scale_of(const MatDesc& d, int mode) {
  const double r = (double)d.rows, c = (double)d.cols;
  if (mode == 1) return 1.f;
  if (mode == 2) return (float)(0.2 * std::sqrt(std::max(r, c)));
  return (float)std::sqrt(std::max(1.0, r / c));
}

cudaEvent_t pool_event(dmuon_ctx* h) {
  if (!h->ev_pool.empty()) { cudaEvent_t e = h->ev_pool.back(); h->ev_pool.pop_back(); return e; }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus c = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &c) == cudaSuccess && c != cudaStreamCaptureStatusNone;
}

struct LaunchGuard {  // brackets one launch with profiling events (not under capture)
  dmuon_ctx* h; cudaStream_t s; ProfRec r; bool on;
  LaunchGuard(dmuon_ctx* h_, cudaStream_t s_, int kind) : h(h_), s(s_), on(h_->profiling && !capturing(s_)) {
    if (on) { r.a = pool_event(h); r.b = pool_event(h); r.kind = kind; cudaEventRecord(r.a, s); }
  }
  ~LaunchGuard() {
    ++h->launches;
    if (on) { cudaEventRecord(r.b, s); h->prof.push_back(r); }
  }
};

int check_ptr(const void* p) {
  if (!p) return DMUON_ERR_ARG;
  if (((uintptr_t)p & 15u) != 0) return DMUON_ERR_ALIGN;
  return DMUON_OK;
}

int check_shapes(const dmuon_shape_t* shapes, int n) {
  for (int i = 0; i < n; ++i) {
    const int64_t r = shapes[i].rows, c = shapes[i].cols;
    if (r <= 0 || c <= 0 || r > DMUON_MAX_DIM || c > DMUON_MAX_DIM) return DMUON_ERR_ARG;
    if (std::min(r, c) > DMUON_MAX_SHORT_SIDE) return DMUON_ERR_ARG;
  }
  return DMUON_OK;
}

// Device buffer for a flat call: host part (descriptors, prefix, bucket
// lists) staged through pinned memory; `dev_extra` bytes of device-only
// scratch follow.  Returns the device base (nullptr on failure).
uint8_t* aux_buffers(dmuon_ctx* h, const std::vector<uint8_t>& host_part, size_t dev_extra,
                     cudaStream_t stream, int* rc) {
  const size_t need = rup((int64_t)host_part.size(), 256) + dev_extra;
  cudaError_t e;
  if (h->aux_dev_cap < need) {
    if (h->aux_dev) {
      e = cudaStreamSynchronize(stream);  // earlier work may still read it
      cudaFree(h->aux_dev);
    }
    h->aux_dev = nullptr;
    h->aux_dev_cap = 0;
    if ((e = cudaMalloc(&h->aux_dev, need)) != cudaSuccess) {
      h->aux_dev = nullptr;
      cudaGetLastError();
      *rc = fail(h, DMUON_ERR_OOM, "aux cudaMalloc", e);
      return nullptr;
    }
    h->aux_dev_cap = need;
  }
  if (h->aux_pending) { cudaEventSynchronize(h->aux_ev); h->aux_pending = false; }
  if (h->aux_host_cap < host_part.size()) {
    if (h->aux_host) cudaFreeHost(h->aux_host);
    h->aux_host = nullptr;
    h->aux_host_cap = 0;
    if (cudaMallocHost(&h->aux_host, host_part.size()) != cudaSuccess) {
      *rc = fail(h, DMUON_ERR_OOM, "aux pinned staging");
      return nullptr;
    }
    h->aux_host_cap = host_part.size();
  }
  std::memcpy(h->aux_host, host_part.data(), host_part.size());
  e = cudaMemcpyAsync(h->aux_dev, h->aux_host, host_part.size(), cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaEventRecord(h->aux_ev, stream);
  if (e != cudaSuccess) {
    *rc = fail(h, cuda_err(e), "aux upload", e);
    return nullptr;
  }
  h->aux_pending = true;
  *rc = DMUON_OK;
  return (uint8_t*)h->aux_dev;
}

// Flat descriptors + tile prefix for a tensor list.
struct FlatPlan {
  std::vector<uint8_t> host;
  size_t off_prefix = 0, off_bstart = 0, off_members = 0;
  int64_t n_tiles = 0;
};

void flat_plan(FlatPlan& fp, const std::vector<FlatDesc>& descs, const std::vector<int>* buckets,
               int n_buckets) {
  const int n = (int)descs.size();
  std::vector<int64_t> prefix(n + 1, 0);
  for (int i = 0; i < n; ++i) prefix[i + 1] = prefix[i] + cdiv(descs[i].numel, kFlatTile);
  fp.n_tiles = prefix[n];
  size_t off = rup(sizeof(FlatDesc) * n, 256);
  fp.off_prefix = off;
  off += rup(8 * (n + 1), 256);
  std::vector<int> bstart, members;
  if (buckets) {
    bstart.assign(n_buckets + 1, 0);
    for (int i = 0; i < n; ++i) ++bstart[(*buckets)[i] + 1];
    for (int b = 0; b < n_buckets; ++b) bstart[b + 1] += bstart[b];
    members.resize(n);
    std::vector<int> fill(bstart.begin(), bstart.end() - 1);
    for (int i = 0; i < n; ++i) members[fill[(*buckets)[i]]++] = i;
    fp.off_bstart = off;
    off += rup(4 * (n_buckets + 1), 256);
    fp.off_members = off;
    off += rup(4 * n, 256);
  }
  fp.host.assign(off, 0);
  std::memcpy(fp.host.data(), descs.data(), sizeof(FlatDesc) * n);
  std::memcpy(fp.host.data() + fp.off_prefix, prefix.data(), 8 * (n + 1));
  if (buckets) {
    std::memcpy(fp.host.data() + fp.off_bstart, bstart.data(), 4 * (n_buckets + 1));
    std::memcpy(fp.host.data() + fp.off_members, members.data(), 4 * n);
  }
}

bool is_vec4(const void* p, int64_t numel) { return (((uintptr_t)p & 15u) == 0) && (numel % 4 == 0); }

// Momentum, Nesterov input, the fp16 iterate X0 = p U and the per-matrix norm
// of a chunk: the momentum pass, the finalisation, then the redo pass and a
// second finalisation for matrices whose prescale p missed its window (both
// return at once when none did).
int run_chunk_norm(dmuon_ctx* h, const Chunk& ch, const MatPtrs* dptrs, float mu, float eps,
                   int nesterov, int ns_only, cudaStream_t stream) {
  const Layout& L = ch.L;
  const int n = ch.n;
  const int64_t nt = L.tile_prefix[n];
  const int grid = (int)std::min<int64_t>(nt, (int64_t)h->num_sms * kMomCtasPerSm);
  cudaError_t e;
  for (int pass = 0; pass < 2; ++pass) {
    {
      MomArgs a{ch.d_mats, dptrs, ch.d_prefix, n, nt, mu, nesterov, ns_only, ch.d_partials, ch.d_tmax,
                ch.d_pscale, ch.d_redo, pass};
      LaunchGuard g(h, stream, DMUON_KIND_MOMENTUM);
      if ((e = launch_mom(a, grid, stream)) != cudaSuccess) return fail(h, cuda_err(e), "mom_norm launch", e);
    }
    {
      FinalizeArgs a{ch.d_mats, ch.d_prefix, ch.d_partials, ch.d_tmax, n, eps, ch.d_svec, ch.d_bvec, ch.d_pscale,
                     ch.d_redo, h->d_flags + ch.i0, pass};
      LaunchGuard g(h, stream, DMUON_KIND_FINALIZE);
      if ((e = launch_finalize(a, stream)) != cudaSuccess) return fail(h, cuda_err(e), "finalize launch", e);
    }
  }
  return DMUON_OK;
}

// Newton-Schulz iterations and the update of a chunk.
int run_chunk_ns(dmuon_ctx* h, const Chunk& ch, const MatPtrs* dptrs, float lr, int ns_steps,
                 const float* coeffs, float wd, int ns_only, cudaStream_t stream) {
  const Layout& L = ch.L;
  const int n = ch.n;
  const int64_t nt = L.tile_prefix[n];
  cudaError_t e;
  const float decay = 1.f - lr * wd;
  if (ns_steps == 0) {
    Update0Args a{ch.d_mats, dptrs, ch.d_prefix, n, nt, ch.d_svec, lr, decay, ns_only};
    const int grid = (int)std::min<int64_t>(nt, (int64_t)h->num_sms * 8);
    LaunchGuard g(h, stream, DMUON_KIND_UPDATE0);
    if ((e = launch_update0(a, grid, stream)) != cudaSuccess) return fail(h, cuda_err(e), "update0 launch", e);
    return DMUON_OK;
  }
  int64_t chunk_items = 0;
  for (int p = 0; p < 3; ++p) chunk_items += (int64_t)L.items[p].size();
  const int avail = h->plan_pair ? h->max_clusters : h->num_sms;
  const bool fuse = h->fused == 1 || (h->fused == 2 && chunk_items <= kFuseItemsPerProc * (int64_t)avail);
  if (fuse && ns_steps <= 64) {
    // One launch for every product of every iteration: each tile waits on its
    // matrix's counter of finished tiles (zeroed here) for the stage before.
    GemmArgs a{};
    a.mats = ch.d_mats;
    a.ptrs = dptrs;
    a.tmaps = ch.d_maps;
    int grid = 0;
    for (int p = 0; p < 3; ++p) {
      a.fitems[p] = ch.d_items[p];
      a.fstarts[p] = L.starts[p].empty() ? nullptr : ch.d_starts[p];
      a.fn_items[p] = (int)L.items[p].size();
      a.fprocs[p] = L.procs[p];
      grid = std::max(grid, L.procs[p]);
    }
    a.n_iters = ns_steps;
    for (int k = 0; k < ns_steps; ++k) {
      const float* row = coeffs ? coeffs + 3 * k : kYouCoefficients[std::min(k, 4)];
      for (int q = 0; q < 3; ++q) a.coef[k][q] = row[q];
    }
    a.counters = ch.d_counters;
    a.f16_iters = h->f16_iters;
    a.fold = 1;
    a.final_mode = ns_only ? kWriteO : kUpdateW;
    a.lr = lr;
    a.decay = decay;
    a.svec = ch.d_svec;
    a.bvec = ch.d_bvec;
    a.err = h->d_err;
    a.timeout_ns = h->wait_timeout_ns;
    if (grid <= 0) return DMUON_OK;
    if ((e = cudaMemsetAsync(ch.d_counters, 0, 4 * (size_t)n, stream)) != cudaSuccess)
      return fail(h, cuda_err(e), "counter reset", e);
    LaunchGuard g(h, stream, DMUON_KIND_NS_FUSED);
    if (h->plan_pair) {
      if ((e = launch_gemm_pair(kPhaseFused, a, grid, stream)) != cudaSuccess)
        return fail(h, cuda_err(e), "ns_gemm_pair fused launch", e);
    } else if ((e = launch_gemm(kPhaseFused, a, grid, stream, h->plan_bn)) != cudaSuccess) {
      return fail(h, cuda_err(e), "ns_gemm fused launch", e);
    }
    return DMUON_OK;
  }
  static const int kKinds[3] = {DMUON_KIND_GRAM, DMUON_KIND_GRAM2, DMUON_KIND_APPLY};
  for (int k = 0; k < ns_steps; ++k) {
    const float* row = coeffs ? coeffs + 3 * k : kYouCoefficients[std::min(k, 4)];
    for (int p = 0; p < 3; ++p) {
      GemmArgs a{};
      a.mats = ch.d_mats;
      a.ptrs = dptrs;
      a.tmaps = ch.d_maps;
      a.items = ch.d_items[p];
      a.starts = L.starts[p].empty() ? nullptr : ch.d_starts[p];
      a.n_items = (int)L.items[p].size();
      a.src = k & 1;
      a.ca = row[0]; a.cb = row[1]; a.cc = row[2];
      a.first = k == 0;
      a.iter = k;
      a.f16_iters = h->f16_iters;
      a.fold = 1;
      a.final_mode = (k == ns_steps - 1) ? (ns_only ? kWriteO : kUpdateW) : kWriteX;
      a.lr = lr;
      a.decay = decay;
      a.svec = ch.d_svec;
      a.bvec = ch.d_bvec;
      a.err = h->d_err;
      a.timeout_ns = h->wait_timeout_ns;
      if (a.n_items <= 0) continue;
      LaunchGuard g(h, stream, kKinds[p]);
      if (h->plan_pair) {
        const int clusters = L.procs[p];  // the processors the list was dealt to
        if ((e = launch_gemm_pair(p, a, clusters, stream)) != cudaSuccess)
          return fail(h, cuda_err(e), "ns_gemm_pair launch", e);
      } else {
        const int grid = L.procs[p];
        if ((e = launch_gemm(p, a, grid, stream, h->plan_bn)) != cudaSuccess)
          return fail(h, cuda_err(e), "ns_gemm launch", e);
      }
    }
  }
  return DMUON_OK;
}


// Newton-Schulz of a chunk with the Gram-space backend and the update.
// Per window: R~ = kappa X X^T, then per step Z (the window's first Q),
// Q' = Z Q (later steps), W~ = R~ Z and R~' = Z W~ (all but the window's last
// step); between windows and at the end the direct Apply kernel forms Q X
// (a = 0), the last one updating W (or writing O).  Windows longer than
// kMaxGramWindow steps are split (restart_windows).
int run_chunk_gram(dmuon_ctx* h, const Chunk& ch, const MatPtrs* dptrs, float lr, int ns_steps,
                   const float* coeffs, float wd, int ns_only, const std::vector<int>& restarts,
                   cudaStream_t stream) {
  const Layout& L = ch.L;
  const int n = ch.n;
  const int64_t nt = L.tile_prefix[n];
  cudaError_t e;
  const float decay = 1.f - lr * wd;
  if (ns_steps == 0) {
    Update0Args a{ch.d_mats, dptrs, ch.d_prefix, n, nt, ch.d_svec, lr, decay, ns_only};
    const int grid = (int)std::min<int64_t>(nt, (int64_t)h->num_sms * 8);
    LaunchGuard g(h, stream, DMUON_KIND_UPDATE0);
    if ((e = launch_update0(a, grid, stream)) != cudaSuccess) return fail(h, cuda_err(e), "update0 launch", e);
    return DMUON_OK;
  }
  const int n_gram = (int)L.items[kPhaseGram].size(), n_prod = (int)L.items[kPhaseGram2].size();
  auto prod = [&](GramArgs a, bool x_operand, int kind) -> int {
    a.gd = ch.d_gd;
    a.mats = ch.d_mats;
    a.xmaps = ch.d_maps;
    a.gmaps = ch.d_gmaps;
    a.x_operand = x_operand ? 1 : 0;
    const int ph = x_operand ? kPhaseGram : kPhaseGram2;
    a.items = ch.d_items[ph];
    a.starts = L.starts[ph].empty() ? nullptr : ch.d_starts[ph];
    a.n_items = x_operand ? n_gram : n_prod;
    a.svec = ch.d_svec;
    a.bvec = ch.d_bvec;
    a.err = h->d_err;
    a.timeout_ns = h->wait_timeout_ns;
    if (a.n_items <= 0) return DMUON_OK;
    LaunchGuard g(h, stream, kind);
    const cudaError_t ee = launch_gram_pair(a, L.procs[ph], stream);
    return ee == cudaSuccess ? DMUON_OK : fail(h, cuda_err(ee), "ns_gram_pair launch", ee);
  };
  auto apply = [&](int src, bool first, int mode) -> int {
    GemmArgs a{};
    a.mats = ch.d_mats;
    a.ptrs = dptrs;
    a.tmaps = ch.d_maps;
    a.items = ch.d_items[kPhaseApply];
    a.starts = L.starts[kPhaseApply].empty() ? nullptr : ch.d_starts[kPhaseApply];
    a.n_items = (int)L.items[kPhaseApply].size();
    a.src = src;
    a.ca = 0.f;          // X' = Q X
    a.f16_iters = 1 << 30;  // the Gram backend is fp16 throughout
    a.fold = 1;          // no a*X term to add: skip reading X in the epilogue
    a.first = first;     // the first window's X is X0 = p U: times s/p
    a.final_mode = mode;
    a.lr = lr;
    a.decay = decay;
    a.svec = ch.d_svec;
    a.bvec = ch.d_bvec;
    a.err = h->d_err;
    a.timeout_ns = h->wait_timeout_ns;
    if (a.n_items <= 0) return DMUON_OK;
    LaunchGuard g(h, stream, DMUON_KIND_APPLY);
    const cudaError_t ee = launch_gemm_pair(kPhaseApply, a, L.procs[kPhaseApply], stream);
    return ee == cudaSuccess ? DMUON_OK : fail(h, cuda_err(ee), "ns_gemm_pair launch", ee);
  };
  auto blank = []() {
    GramArgs a{};
    a.out2 = a.add1 = -1;
    a.g0 = 1.f;
    return a;
  };
  const auto windows = restart_windows(ns_steps, restarts);
  int rc;
  // One window of steps [k0, k1): per step Z (into Z0 / Z1 alternately),
  // Q' = Z Q from the second step on (the first step's Q is its Z, read
  // from that Z buffer), and, unless it is the window's last step, W = R Z
  // and R' = Z W.  The window's final factor goes to kGbQb (a one-step
  // window writes its Z there too); Q' products of earlier steps alternate
  // between Q0 and Q1.
  auto window = [&](int k0, int k1) -> int {
    int rc_ = kGbR0, zc = kGbZ0, qc = -1;
    for (int k = k0; k < k1; ++k) {
      const float* row = coeffs ? coeffs + 3 * k : kYouCoefficients[std::min(k, 4)];
      const bool wfirst = k == k0, wlast = k == k1 - 1;
      {  // Z = a I + (b/kappa) R~ + (c/kappa^2) R~ R~
        GramArgs a = blank();
        a.opA = a.opB = rc_;
        a.out = zc;
        a.g0 = row[2];
        a.gpow = -2;
        a.add1 = rc_;
        a.c1 = row[1];
        a.p1pow = -1;
        a.diag = row[0];
        if (wfirst && wlast) a.out2 = kGbQb;
        if ((rc = prod(a, false, DMUON_KIND_GS_PROD))) return rc;
      }
      if (!wfirst) {  // Q' = Z Q
        GramArgs a = blank();
        a.opA = zc;
        a.opB = qc;
        a.out = wlast ? kGbQb : (qc == kGbQ0 ? kGbQ1 : kGbQ0);
        if ((rc = prod(a, false, DMUON_KIND_GS_PROD))) return rc;
        qc = a.out;
      } else {
        qc = zc;  // Q of the first step is its Z
      }
      if (!wlast) {
        GramArgs a = blank();  // W~ = R~ Z
        a.opA = rc_;
        a.opB = zc;
        a.out = kGbW;
        if ((rc = prod(a, false, DMUON_KIND_GS_PROD))) return rc;
        GramArgs r = blank();  // R~' = Z W~
        r.opA = zc;
        r.opB = kGbW;
        r.out = rc_ ^ kGbR0 ^ kGbR1;
        if ((rc = prod(r, false, DMUON_KIND_GS_PROD))) return rc;
        rc_ ^= kGbR0 ^ kGbR1;
      }
      zc = zc == kGbZ0 ? kGbZ1 : kGbZ0;
    }
    return DMUON_OK;
  };
  int src = 0;
  bool first = true;
  for (size_t wi = 0; wi < windows.size(); ++wi) {
    if (wi > 0) {  // restart: X <- Q X, then a new window from the explicit iterate
      if ((rc = apply(src, first, kWriteX))) return rc;
      src ^= 1;
      first = false;
    }
    {  // R~ = kappa X X^T of the true X: (s/p)^2 on the first window's X0 = p U, 1/beta^2 after
      GramArgs a = blank();
      a.src = src;
      a.out = kGbR0;
      a.gpow = 1;
      a.xscale = first ? 1 : 2;
      if ((rc = prod(a, true, DMUON_KIND_GS_GRAM))) return rc;
    }
    if ((rc = window(windows[wi].first, windows[wi].second))) return rc;
  }
  return apply(src, first, ns_only ? kWriteO : kUpdateW);
}

// Shared by dmuon_step (ns_only = 0) and dmuon_newton_schulz (ns_only = 1).
int run(dmuon_ctx* h, const MatPtrs* ptrs, const dmuon_shape_t* shapes, int n, float lr, float mu,
        int ns_steps, const float* coeffs, float eps, float wd, int nesterov, int scale_mode,
        int ns_only, cudaStream_t stream, bool gram = false, const std::vector<int>& restarts = {}) {
  if (cudaSetDevice(h->device) != cudaSuccess) return fail(h, DMUON_ERR_CUDA, "cudaSetDevice");
  // Under stream capture nothing may allocate, upload or synchronise: the
  // plan, the update scales and the pointer set must already exist from an
  // earlier call with the same shapes, options and buffers.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return fail(h, DMUON_ERR_CUDA, "cudaStreamIsCapturing");
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  if (capturing && !same_shapes(h, shapes, n, gram))
    return fail(h, DMUON_ERR_ARG, "stream capture: call once with these shapes before capturing");
  int rc = build_plan(h, shapes, n, gram);
  if (rc) return rc;

  // Per-matrix update scale depends on the mode: refresh descriptors when
  // it changes (rare; synchronous copy of small arrays).
  cudaError_t e = cudaSuccess;
  for (Chunk& ch : h->chunks) {
    bool dirty = false;
    for (int i = 0; i < ch.n; ++i) {
      const float s = scale_of(ch.L.mats[i], scale_mode);
      if (ch.L.mats[i].scale != s) { ch.L.mats[i].scale = s; dirty = true; }
    }
    if (dirty && capturing)
      return fail(h, DMUON_ERR_ARG, "stream capture: call once with this scale_mode before capturing");
    if (dirty) {
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaMemcpy(ch.d_mats, ch.L.mats.data(), sizeof(MatDesc) * ch.n, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return fail(h, cuda_err(e), "descriptor refresh", e);
    }
  }
  {
    bool dirty = false;
    for (SmallDesc& d : h->small_descs) {
      MatDesc md{};
      md.rows = d.rows;
      md.cols = d.cols;
      const float s = scale_of(md, scale_mode);
      if (d.scale != s) { d.scale = s; dirty = true; }
    }
    if (dirty && capturing)
      return fail(h, DMUON_ERR_ARG, "stream capture: call once with this scale_mode before capturing");
    if (dirty) {
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess)
        e = cudaMemcpy(h->d_small, h->small_descs.data(), sizeof(SmallDesc) * h->small_descs.size(),
                       cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return fail(h, cuda_err(e), "descriptor refresh", e);
    }
  }

  // Caller pointer sets are cached in kPtrSlots device slots (least recently
  // used is replaced), so alternating between a few lists of buffers -- e.g.
  // one call per layer -- uploads nothing after the first round.
  int slot = -1;
  for (int k = 0; k < kPtrSlots && slot < 0; ++k) {
    const std::vector<MatPtrs>& sp = h->slot_ptrs[k];
    if ((int)sp.size() != n) continue;
    bool same = true;
    for (int i = 0; same && i < n; ++i)
      same = sp[i].W == ptrs[i].W && sp[i].G == ptrs[i].G && sp[i].M == ptrs[i].M;
    if (same) slot = k;
  }
  if (slot < 0 && capturing)
    return fail(h, DMUON_ERR_ARG, "stream capture: call once with these buffers before capturing");
  if (slot < 0) {
    slot = 0;
    for (int k = 1; k < kPtrSlots; ++k)
      if (h->slot_use[k] < h->slot_use[slot]) slot = k;
    // The slot's pinned staging may still feed an earlier copy.
    if (h->slot_pending[slot]) { cudaEventSynchronize(h->slot_ev[slot]); h->slot_pending[slot] = false; }
    MatPtrs* stage = h->h_stage + (size_t)slot * n;
    for (int k = 0; k < n; ++k) stage[k] = ptrs[h->order[k]];  // plan order
    e = cudaMemcpyAsync(h->d_ptrs + (size_t)slot * n, stage, sizeof(MatPtrs) * n, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaEventRecord(h->slot_ev[slot], stream);
    if (e != cudaSuccess) return fail(h, cuda_err(e), "pointer upload", e);
    h->slot_pending[slot] = true;
    h->slot_ptrs[slot].assign(ptrs, ptrs + n);
  }
  h->slot_use[slot] = ++h->use_clock;
  const MatPtrs* dptrs = h->d_ptrs + (size_t)slot * n;
  h->last_stream = stream;

  if (!h->small_descs.empty()) {
    SmallArgs a{};
    a.descs = h->d_small;
    a.ptrs = dptrs;
    a.flags = h->d_flags;
    a.err = h->d_err;
    a.timeout_ns = h->wait_timeout_ns;
    a.ns_steps = ns_steps;
    a.ns_only = ns_only;
    a.nesterov = nesterov;
    a.mu = mu;
    a.eps = eps;
    a.lr = lr;
    a.decay = 1.f - lr * wd;
    for (int k = 0; k < ns_steps; ++k) {
      const float* row = coeffs ? coeffs + 3 * k : kYouCoefficients[std::min(k, 4)];
      for (int q = 0; q < 3; ++q) a.coeffs[k][q] = row[q];
    }
    LaunchGuard g(h, stream, DMUON_KIND_SMALL);
    if ((e = launch_small(a, (int)h->small_descs.size(), stream)) != cudaSuccess)
      return fail(h, cuda_err(e), "ns_small launch", e);
  }

  auto chunk_ns = [&](const Chunk& ch, cudaStream_t st) {
    return h->plan_gram ? run_chunk_gram(h, ch, dptrs + ch.i0, lr, ns_steps, coeffs, wd, ns_only, restarts, st)
                        : run_chunk_ns(h, ch, dptrs + ch.i0, lr, ns_steps, coeffs, wd, ns_only, st);
  };
  if (!h->plan_overlap) {
    for (const Chunk& ch : h->chunks) {
      if ((rc = run_chunk_norm(h, ch, dptrs + ch.i0, mu, eps, nesterov, ns_only, stream))) return rc;
      if ((rc = chunk_ns(ch, stream))) return rc;
    }
    return DMUON_OK;
  }
  // Chunk c's momentum pass runs on the side stream into workspace c % 2
  // once chunk c-2's tensor-core phases (same workspace) are done; chunk c's
  // phases run on the caller's stream once its norm is ready.  Enqueued
  // chunk by chunk so every event is recorded before it is waited on.
  if ((e = cudaEventRecord(h->ev_fork, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(h->side, h->ev_fork, 0)) != cudaSuccess)
    return fail(h, cuda_err(e), "overlap fork", e);
  for (size_t c = 0; c < h->chunks.size(); ++c) {
    const Chunk& ch = h->chunks[c];
    const int b = (int)(c & 1);
    if (c >= 2 && (e = cudaStreamWaitEvent(h->side, h->ev_gemm[b], 0)) != cudaSuccess)
      return fail(h, cuda_err(e), "overlap wait", e);
    if ((rc = run_chunk_norm(h, ch, dptrs + ch.i0, mu, eps, nesterov, ns_only, h->side))) return rc;
    if ((e = cudaEventRecord(h->ev_norm[b], h->side)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, h->ev_norm[b], 0)) != cudaSuccess)
      return fail(h, cuda_err(e), "overlap hand-off", e);
    if ((rc = chunk_ns(ch, stream))) return rc;
    if ((e = cudaEventRecord(h->ev_gemm[b], stream)) != cudaSuccess)
      return fail(h, cuda_err(e), "overlap record", e);
  }
  if ((e = cudaEventRecord(h->ev_join, h->side)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, h->ev_join, 0)) != cudaSuccess)
    return fail(h, cuda_err(e), "overlap join", e);
  return DMUON_OK;
}

bool finite3(const float* c, int rows) {
  for (int i = 0; i < 3 * rows; ++i)
    if (!std::isfinite(c[i])) return false;
  return true;
}

// The Gram-space backend's default coefficients ("API Reference", sections
// gram_newton_schulz and POLAR_EXPRESS_COEFFICIENTS: Polar Express with the
// safety factor 1.05): the table dmuon_polar_express_coefficients derives
// from [1e-3, 1], cached per step count.  nullptr if the derivation fails.
const float* gram_default_table(int ns_steps) {
  static std::mutex mu;
  static std::vector<float> cache[DMUON_MAX_NS_STEPS + 1];
  if (ns_steps <= 0 || ns_steps > DMUON_MAX_NS_STEPS) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  std::vector<float>& v = cache[ns_steps];
  if (v.empty()) {
    v.resize(3 * (size_t)ns_steps);
    if (dmuon_polar_express_coefficients(ns_steps, 1e-3, 1.0, 1.05, v.data()) != DMUON_OK) v.clear();
  }
  return v.empty() ? nullptr : v.data();
}

// The direct iteration's fp16 range check of the coefficient table
// (direct_table_fits).
int direct_options(dmuon_ctx* h, int ns_steps, const float* coeffs) {
  char why[192];
  if (!direct_table_fits(ns_steps, coeffs, why, sizeof why)) {
    std::string msg = std::string("coefficient table: ") + why;
    return fail(h, DMUON_ERR_ARG, msg.c_str());
  }
  return DMUON_OK;
}

// Gram-space backend: the coefficient table (NULL = its Polar Express
// default, returned in *table), restart positions (NULL = the pages' default
// {2}) and the fp16 range check (gram_table_fits).
int gram_options(dmuon_ctx* h, int ns_steps, const float* coeffs, const int* restarts, int n_restarts,
                 std::vector<int>* out, const float** table) {
  *table = coeffs;
  if (!coeffs && ns_steps > 0) {
    *table = gram_default_table(ns_steps);
    if (!*table) return fail(h, DMUON_ERR_ARG, "Gram-space backend: Polar Express table derivation failed");
  }
  coeffs = *table;
  out->clear();
  if (!restarts) {
    out->push_back(2);
  } else {
    if (n_restarts < 0 || n_restarts > DMUON_MAX_NS_STEPS) return fail(h, DMUON_ERR_ARG, "n_restarts out of range");
    out->assign(restarts, restarts + n_restarts);
  }
  char why[192];
  if (!gram_table_fits(ns_steps, coeffs, *out, why, sizeof why)) {
    std::string msg = std::string("Gram-space backend: ") + why;
    return fail(h, DMUON_ERR_ARG, msg.c_str());
  }
  return DMUON_OK;
}

}  // namespace

extern "C" {

void dmuon_default_opts(dmuon_opts_t* o) {
  if (!o) return;
  o->weight_decay = 0.f;
  o->eps = 1e-7f;
  o->nesterov = 1;
  o->scale_mode = 0;
  o->coeffs = nullptr;
  o->backend = DMUON_BACKEND_DIRECT;
  o->restarts = nullptr;
  o->n_restarts = 0;
}

int dmuon_create(dmuon_handle_t* out, int device) {
  if (!out) return DMUON_ERR_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess) { cudaGetLastError(); return DMUON_ERR_CUDA; }
  if (device < 0 || device >= count) return DMUON_ERR_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return DMUON_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (major != 10 || minor != 3) return DMUON_ERR_UNSUPPORTED;
  if (gemm_configure() != cudaSuccess) return DMUON_ERR_CUDA;
  const bool small_ok = small_configure() == cudaSuccess;
  if (!small_ok) cudaGetLastError();
  int clusters = 0;
  if (gemm_pair_configure(&clusters) != cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  const bool gram_ok = clusters > 0 && gram_configure() == cudaSuccess;
  if (!gram_ok) cudaGetLastError();
  dmuon_ctx* h = new dmuon_ctx();
  h->device = device;
  h->num_sms = sms;
  h->max_clusters = clusters;
  h->small_ok = small_ok;
  h->gram_ok = gram_ok;
  for (int k = 0; k < kPtrSlots; ++k) {
    if (cudaEventCreateWithFlags(&h->slot_ev[k], cudaEventDisableTiming) != cudaSuccess) {
      for (int j = 0; j < k; ++j) cudaEventDestroy(h->slot_ev[j]);
      delete h;
      return DMUON_ERR_CUDA;
    }
  }
  if (cudaEventCreateWithFlags(&h->aux_ev, cudaEventDisableTiming) != cudaSuccess) {
    for (int k = 0; k < kPtrSlots; ++k) cudaEventDestroy(h->slot_ev[k]);
    delete h;
    return DMUON_ERR_CUDA;
  }
  bool ok = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) == cudaSuccess;
  for (int b = 0; b < 2; ++b) {
    ok = ok && cudaEventCreateWithFlags(&h->ev_norm[b], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&h->ev_gemm[b], cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    dmuon_destroy(h);
    return DMUON_ERR_CUDA;
  }
  *out = h;
  return DMUON_OK;
}

void dmuon_destroy(dmuon_handle_t h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_plan(h);
  for (int k = 0; k < kPtrSlots; ++k)
    if (h->slot_ev[k]) cudaEventDestroy(h->slot_ev[k]);
  if (h->aux_ev) cudaEventDestroy(h->aux_ev);
  for (cudaEvent_t ev : {h->ev_fork, h->ev_join, h->ev_norm[0], h->ev_norm[1], h->ev_gemm[0], h->ev_gemm[1]})
    if (ev) cudaEventDestroy(ev);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->aux_dev) cudaFree(h->aux_dev);
  if (h->aux_host) cudaFreeHost(h->aux_host);
  for (auto& r : h->prof) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
  for (auto e : h->ev_pool) cudaEventDestroy(e);
  delete h;
}

int dmuon_workspace_bytes(const dmuon_shape_t* shapes, int n_mats, size_t* out_bytes) {
  if (!out_bytes || n_mats < 0 || (n_mats > 0 && !shapes)) return DMUON_ERR_ARG;
  *out_bytes = 0;
  if (n_mats == 0) return DMUON_OK;
  if (int rc = check_shapes(shapes, n_mats)) return rc;
  // The largest plan over tile kinds, with and without the small-matrix
  // kernel (which needs no workspace).
  size_t most = 0;
  for (int kind = 0; kind < 3; ++kind)  // single CTAs 128 x 256, CTA pairs, single CTAs 128 x 128
    for (int sp = 0; sp < 2; ++sp) {
      size_t ws, sm;
      plan_sizes(shapes, n_mats, kind == 1, kDefaultChunkElems, sp != 0, &ws, &sm, false, kind == 2 ? kBM : kBN);
      most = std::max(most, ws + sm);
    }
  *out_bytes = most;
  return DMUON_OK;
}

int dmuon_workspace_bytes_ex(const dmuon_shape_t* shapes, int n_mats, int backend, size_t* out_bytes) {
  if (backend == DMUON_BACKEND_DIRECT) return dmuon_workspace_bytes(shapes, n_mats, out_bytes);
  if (backend != DMUON_BACKEND_GRAM || !out_bytes || n_mats < 0 || (n_mats > 0 && !shapes)) return DMUON_ERR_ARG;
  *out_bytes = 0;
  if (n_mats == 0) return DMUON_OK;
  if (int rc = check_shapes(shapes, n_mats)) return rc;
  size_t most = 0;
  for (int sp = 0; sp < 2; ++sp) {
    size_t ws, sm;
    plan_sizes(shapes, n_mats, true, kDefaultChunkElems, sp != 0, &ws, &sm, true);
    most = std::max(most, ws + sm);
  }
  *out_bytes = most;
  return DMUON_OK;
}

int dmuon_step(dmuon_handle_t h, float* const* params, const float* const* grads,
               float* const* momentum, const dmuon_shape_t* shapes, int n_mats, float lr,
               float mu, int ns_steps, const dmuon_opts_t* opts, void* stream) {
  if (!h || n_mats < 0) return DMUON_ERR_ARG;
  if (n_mats == 0) return DMUON_OK;
  if (!params || !grads || !momentum || !shapes) return DMUON_ERR_ARG;
  if (ns_steps < 0 || ns_steps > DMUON_MAX_NS_STEPS) return DMUON_ERR_ARG;
  if (!std::isfinite(lr) || !std::isfinite(mu)) return DMUON_ERR_ARG;
  dmuon_opts_t o;
  dmuon_default_opts(&o);
  if (opts) o = *opts;
  if (!std::isfinite(o.weight_decay) || !std::isfinite(o.eps) || o.eps < 0.f) return DMUON_ERR_ARG;
  if (o.scale_mode < 0 || o.scale_mode > 2) return DMUON_ERR_ARG;
  if (o.coeffs && !finite3(o.coeffs, ns_steps)) return DMUON_ERR_ARG;
  if (o.backend != DMUON_BACKEND_DIRECT && o.backend != DMUON_BACKEND_GRAM) return DMUON_ERR_ARG;
  if (int rc = check_shapes(shapes, n_mats)) return rc;
  std::vector<int> restarts;
  const float* table = o.coeffs;
  if (o.backend == DMUON_BACKEND_GRAM) {
    if (int rc = gram_options(h, ns_steps, o.coeffs, o.restarts, o.n_restarts, &restarts, &table)) return rc;
  } else if (int rc = direct_options(h, ns_steps, o.coeffs)) {
    return rc;
  }
  std::vector<MatPtrs> ptrs(n_mats);
  for (int i = 0; i < n_mats; ++i) {
    int rc;
    if ((rc = check_ptr(params[i])) || (rc = check_ptr(grads[i])) || (rc = check_ptr(momentum[i]))) return rc;
    if ((const void*)params[i] == (const void*)grads[i] || params[i] == momentum[i] ||
        (const void*)grads[i] == (const void*)momentum[i])
      return DMUON_ERR_ARG;
    ptrs[i] = MatPtrs{params[i], grads[i], momentum[i], nullptr};
  }
  return run(h, ptrs.data(), shapes, n_mats, lr, mu, ns_steps, table, o.eps, o.weight_decay,
             o.nesterov ? 1 : 0, o.scale_mode, 0, (cudaStream_t)stream, o.backend == DMUON_BACKEND_GRAM, restarts);
}

int dmuon_newton_schulz(dmuon_handle_t h, const float* const* inputs, float* const* outputs,
                        const dmuon_shape_t* shapes, int n_mats, int ns_steps, const float* coeffs,
                        float eps, void* stream) {
  if (!h || n_mats < 0) return DMUON_ERR_ARG;
  if (n_mats == 0) return DMUON_OK;
  if (!inputs || !outputs || !shapes) return DMUON_ERR_ARG;
  if (ns_steps < 0 || ns_steps > DMUON_MAX_NS_STEPS) return DMUON_ERR_ARG;
  if (!std::isfinite(eps)) return DMUON_ERR_ARG;
  if (eps <= 0.f) eps = 1e-7f;
  if (coeffs && !finite3(coeffs, ns_steps)) return DMUON_ERR_ARG;
  if (int rc = check_shapes(shapes, n_mats)) return rc;
  if (int rc = direct_options(h, ns_steps, coeffs)) return rc;
  std::vector<MatPtrs> ptrs(n_mats);
  for (int i = 0; i < n_mats; ++i) {
    int rc;
    if ((rc = check_ptr(inputs[i])) || (rc = check_ptr(outputs[i]))) return rc;
    if ((const void*)inputs[i] == (const void*)outputs[i]) return DMUON_ERR_ARG;
    ptrs[i] = MatPtrs{outputs[i], inputs[i], nullptr, nullptr};
  }
  return run(h, ptrs.data(), shapes, n_mats, 0.f, 0.f, ns_steps, coeffs, eps, 0.f, 0, 1, 1,
             (cudaStream_t)stream);
}

int dmuon_gram_newton_schulz(dmuon_handle_t h, const float* const* inputs, float* const* outputs,
                             const dmuon_shape_t* shapes, int n_mats, int ns_steps, const float* coeffs,
                             const int* restarts, int n_restarts, float eps, void* stream) {
  if (!h || n_mats < 0) return DMUON_ERR_ARG;
  if (n_mats == 0) return DMUON_OK;
  if (!inputs || !outputs || !shapes) return DMUON_ERR_ARG;
  if (ns_steps < 0 || ns_steps > DMUON_MAX_NS_STEPS) return DMUON_ERR_ARG;
  if (!std::isfinite(eps)) return DMUON_ERR_ARG;
  if (eps <= 0.f) eps = 1e-7f;
  if (coeffs && !finite3(coeffs, ns_steps)) return DMUON_ERR_ARG;
  if (int rc = check_shapes(shapes, n_mats)) return rc;
  std::vector<int> rs;
  const float* table = coeffs;
  if (int rc = gram_options(h, ns_steps, coeffs, restarts, n_restarts, &rs, &table)) return rc;
  std::vector<MatPtrs> ptrs(n_mats);
  for (int i = 0; i < n_mats; ++i) {
    int rc;
    if ((rc = check_ptr(inputs[i])) || (rc = check_ptr(outputs[i]))) return rc;
    if ((const void*)inputs[i] == (const void*)outputs[i]) return DMUON_ERR_ARG;
    ptrs[i] = MatPtrs{outputs[i], inputs[i], nullptr, nullptr};
  }
  return run(h, ptrs.data(), shapes, n_mats, 0.f, 0.f, ns_steps, table, eps, 0.f, 0, 1, 1,
             (cudaStream_t)stream, true, rs);
}

int dmuon_adamw_step(dmuon_handle_t h, float* const* params, const float* const* grads,
                     float* const* exp_avg, float* const* exp_avg_sq, const int64_t* numels, int n,
                     float lr, float beta1, float beta2, float eps, float weight_decay, int step,
                     void* stream_) {
  if (!h || n < 0) return DMUON_ERR_ARG;
  if (n == 0) return DMUON_OK;
  if (!params || !grads || !exp_avg || !exp_avg_sq || !numels) return DMUON_ERR_ARG;
  if (step < 1 || !std::isfinite(lr) || !std::isfinite(beta1) || !std::isfinite(beta2) ||
      !std::isfinite(eps) || !std::isfinite(weight_decay) || beta1 < 0.f || beta1 >= 1.f ||
      beta2 < 0.f || beta2 >= 1.f)
    return DMUON_ERR_ARG;
  std::vector<FlatDesc> descs(n);
  for (int i = 0; i < n; ++i) {
    const void* ps[4] = {params[i], grads[i], exp_avg[i], exp_avg_sq[i]};
    if (numels[i] <= 0) return DMUON_ERR_ARG;
    for (int k = 0; k < 4; ++k) {
      if (!ps[k]) return DMUON_ERR_ARG;
      if ((uintptr_t)ps[k] & 3u) return DMUON_ERR_ALIGN;
      for (int j = 0; j < k; ++j)
        if (ps[j] == ps[k]) return DMUON_ERR_ARG;
    }
    bool v4 = true;
    for (int k = 0; k < 4; ++k) v4 = v4 && is_vec4(ps[k], numels[i]);
    descs[i] = FlatDesc{params[i], grads[i], exp_avg[i], exp_avg_sq[i], numels[i], 0, v4 ? 1 : 0};
  }
  if (cudaSetDevice(h->device) != cudaSuccess) return fail(h, DMUON_ERR_CUDA, "cudaSetDevice");
  cudaStream_t stream = (cudaStream_t)stream_;
  FlatPlan fp;
  flat_plan(fp, descs, nullptr, 0);
  int rc;
  uint8_t* base = aux_buffers(h, fp.host, 0, stream, &rc);
  if (!base) return rc;
  AdamWArgs a{};
  a.descs = (const FlatDesc*)base;
  a.tile_prefix = (const int64_t*)(base + fp.off_prefix);
  a.n = n;
  a.n_tiles = fp.n_tiles;
  a.decay = 1.f - lr * weight_decay;
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.step_size = (float)((double)lr / (1.0 - std::pow((double)beta1, step)));
  a.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(1.0 - std::pow((double)beta2, step)));
  a.eps = eps;
  const int grid = (int)std::min<int64_t>(fp.n_tiles, (int64_t)h->num_sms * 8);
  LaunchGuard g(h, stream, DMUON_KIND_ADAMW);
  cudaError_t e = launch_adamw(a, grid, stream);
  if (e != cudaSuccess) return fail(h, cuda_err(e), "adamw launch", e);
  h->last_stream = stream;
  return DMUON_OK;
}

int dmuon_clip_grad_norm(dmuon_handle_t h, float* const* grads, const int64_t* numels, int n,
                         const int* buckets, int n_buckets, float max_norm, float* norms_out,
                         float* coefs_out, void* stream_) {
  if (!h || n < 0) return DMUON_ERR_ARG;
  if (!buckets) n_buckets = 1;
  if (n_buckets < 1 || !std::isfinite(max_norm)) return DMUON_ERR_ARG;
  if (n == 0) {
    for (int b = 0; b < n_buckets; ++b) {
      if (norms_out) norms_out[b] = 0.f;
      if (coefs_out) coefs_out[b] = max_norm > 0.f ? (float)(max_norm / 1e-6) : -1.f;
    }
    return DMUON_OK;
  }
  if (!grads || !numels) return DMUON_ERR_ARG;
  std::vector<FlatDesc> descs(n);
  std::vector<int> bk(n, 0);
  for (int i = 0; i < n; ++i) {
    if (!grads[i] || numels[i] <= 0) return DMUON_ERR_ARG;
    if ((uintptr_t)grads[i] & 3u) return DMUON_ERR_ALIGN;
    if (buckets) {
      if (buckets[i] < 0 || buckets[i] >= n_buckets) return DMUON_ERR_ARG;
      bk[i] = buckets[i];
    }
    descs[i] = FlatDesc{nullptr, grads[i], nullptr, nullptr, numels[i], bk[i],
                        is_vec4(grads[i], numels[i]) ? 1 : 0};
  }
  if (cudaSetDevice(h->device) != cudaSuccess) return fail(h, DMUON_ERR_CUDA, "cudaSetDevice");
  cudaStream_t stream = (cudaStream_t)stream_;
  FlatPlan fp;
  flat_plan(fp, descs, &bk, n_buckets);
  const size_t off_part = rup((int64_t)fp.host.size(), 256);
  const size_t off_norms = off_part + rup(4 * fp.n_tiles, 256);
  const size_t off_coefs = off_norms + rup(4 * n_buckets, 256);
  const size_t extra = off_coefs + rup(4 * n_buckets, 256) - off_part;
  int rc;
  uint8_t* base = aux_buffers(h, fp.host, extra, stream, &rc);
  if (!base) return rc;
  ClipArgs a{};
  a.descs = (const FlatDesc*)base;
  a.tile_prefix = (const int64_t*)(base + fp.off_prefix);
  a.n = n;
  a.n_tiles = fp.n_tiles;
  a.bucket_start = (const int*)(base + fp.off_bstart);
  a.bucket_members = (const int*)(base + fp.off_members);
  a.n_buckets = n_buckets;
  a.max_norm = max_norm;
  a.partials = (float*)(base + off_part);
  a.norms = (float*)(base + off_norms);
  a.coefs = (float*)(base + off_coefs);
  const int grid = (int)std::min<int64_t>(fp.n_tiles, (int64_t)h->num_sms * 8);
  cudaError_t e;
  {
    LaunchGuard g(h, stream, DMUON_KIND_CLIP);
    h->launches += max_norm > 0.f ? 2 : 1;  // sum of squares, finalise, (scale)
    if ((e = launch_clip(a, grid, stream)) != cudaSuccess) return fail(h, cuda_err(e), "clip launch", e);
  }
  h->last_stream = stream;
  if (norms_out || coefs_out) {
    std::vector<float> nb(n_buckets), cb(n_buckets);
    e = cudaMemcpyAsync(nb.data(), a.norms, 4 * n_buckets, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(cb.data(), a.coefs, 4 * n_buckets, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(h, cuda_err(e), "clip readback", e);
    for (int b = 0; b < n_buckets; ++b) {
      if (norms_out) norms_out[b] = nb[b];
      if (coefs_out) coefs_out[b] = cb[b];
    }
  }
  return DMUON_OK;
}

int dmuon_get_status(dmuon_handle_t h, int* flags, int n_flags) {
  if (!h || n_flags < 0) return DMUON_ERR_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return DMUON_ERR_CUDA;
  cudaError_t e = h->last_stream ? cudaStreamSynchronize(h->last_stream) : cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(h, DMUON_ERR_CUDA, "stream synchronize", e);
  if (!h->small) return DMUON_OK;
  const int n = (int)h->shapes.size();
  std::vector<int> f(n, 0);
  int err = 0;
  std::vector<int> fp(n, 0);
  e = cudaMemcpy(fp.data(), h->d_flags, 4 * n, cudaMemcpyDeviceToHost);
  for (int k = 0; k < n; ++k) f[h->order[k]] = fp[k];  // plan order -> caller order
  if (e == cudaSuccess) e = cudaMemcpy(&err, h->d_err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->d_flags, 0, 4 * n);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, 4);
  if (e != cudaSuccess) return DMUON_ERR_CUDA;
  if (flags)
    for (int i = 0; i < std::min(n, n_flags); ++i) flags[i] = f[i];
  if (err) return DMUON_ERR_TIMEOUT;
  for (int i = 0; i < n; ++i)
    if (f[i]) return DMUON_ERR_NONFINITE;
  return DMUON_OK;
}

int64_t dmuon_launch_count(dmuon_handle_t h) { return h ? h->launches : -1; }

const char* dmuon_last_error(dmuon_handle_t h) {
  if (!h) return "null handle";
  return h->last_error.c_str();
}

int dmuon_set_wait_timeout(dmuon_handle_t h, uint64_t ns) {
  if (!h) return DMUON_ERR_ARG;
  h->wait_timeout_ns = ns;
  return DMUON_OK;
}

int dmuon_set_chunk_elements(dmuon_handle_t h, int64_t elems) {
  if (!h || elems < 0) return DMUON_ERR_ARG;
  h->chunk_elems = elems;
  return DMUON_OK;
}

int dmuon_set_overlap(dmuon_handle_t h, int on) {
  if (!h) return DMUON_ERR_ARG;
  h->overlap = on != 0;
  return DMUON_OK;
}

int dmuon_set_balanced_dealing(dmuon_handle_t h, int on) {
  if (!h) return DMUON_ERR_ARG;
  h->balanced = on != 0;
  return DMUON_OK;
}

int dmuon_set_fp16_iterations(dmuon_handle_t h, int iters) {
  if (!h || iters < 1) return DMUON_ERR_ARG;
  h->f16_iters = iters;
  return DMUON_OK;
}

int dmuon_set_fused_phases(dmuon_handle_t h, int mode) {
  if (!h || mode < 0 || mode > 2) return DMUON_ERR_ARG;
  h->fused = mode;
  return DMUON_OK;
}

int dmuon_set_small_path(dmuon_handle_t h, int on) {
  if (!h) return DMUON_ERR_ARG;
  if (on && !h->small_ok) return DMUON_ERR_UNSUPPORTED;
  h->small_path = on != 0;
  return DMUON_OK;
}

int dmuon_set_tile_mode(dmuon_handle_t h, int mode) {
  if (!h || mode < 0 || mode > 3) return DMUON_ERR_ARG;
  if (mode == 2 && h->max_clusters <= 0) return DMUON_ERR_UNSUPPORTED;
  h->tile_mode = mode;
  return DMUON_OK;
}

int dmuon_profile_enable(dmuon_handle_t h, int on) {
  if (!h) return DMUON_ERR_ARG;
  h->profiling = on != 0;
  return DMUON_OK;
}

int dmuon_profile_read(dmuon_handle_t h, double* ms, int64_t* count, int n_kinds) {
  if (!h || n_kinds < 0 || (n_kinds > 0 && (!ms || !count))) return DMUON_ERR_ARG;
  int rc = DMUON_OK;
  for (auto& r : h->prof) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = DMUON_ERR_CUDA;
    if (r.kind < n_kinds) { ms[r.kind] += t; count[r.kind] += 1; }
    h->ev_pool.push_back(r.a);
    h->ev_pool.push_back(r.b);
  }
  h->prof.clear();
  return rc;
}

int dmuon_plan_summary(dmuon_handle_t h, char* buf, size_t len) {
  if (!h) return DMUON_ERR_ARG;
  std::string s;
  char line[384];
  const int n = (int)h->shapes.size();
  std::snprintf(line, sizeof line, "device %d, %d SMs, %d 2-CTA clusters; matrices %d; backend %s; tiles %s; ",
                h->device, h->num_sms, h->max_clusters, n, h->plan_gram ? "gram" : "direct",
                h->plan_pair ? "256x256 CTA pairs" : (h->plan_bn == kBM ? "128x128 single CTAs" : "128x256 single CTAs"));
  s += line;
  if (h->small) {
    int64_t tiles = 0;
    size_t it[3] = {0, 0, 0};
    for (const Chunk& ch : h->chunks) {
      tiles += ch.L.tile_prefix[ch.n];
      for (int q = 0; q < 3; ++q) it[q] += ch.L.items[q].size();
    }
    // Dealing quality per phase: the busiest processor's item cost over the
    // mean cost per processor, summed over chunks (1 = perfectly even).
    double busiest[3] = {0, 0, 0}, mean[3] = {0, 0, 0};
    for (const Chunk& ch : h->chunks)
      for (int q = 0; q < 3; ++q) {
        const auto b = deal_balance(ch.L, q);
        busiest[q] += b.first;
        mean[q] += b.second;
      }
    double bal[3];
    for (int q = 0; q < 3; ++q) bal[q] = mean[q] > 0 ? busiest[q] / mean[q] : 1.0;
    std::snprintf(line, sizeof line,
                  "small-matrix kernel %zu; chunks %zu (<= %lld elements); momentum tiles %lld; "
                  "items gram %zu gram2 %zu apply %zu; balance gram %.4f gram2 %.4f apply %.4f; "
                  "workspace %.3f GB + %.3f MB",
                  h->small_descs.size(), h->chunks.size(), (long long)h->plan_chunk_elems, (long long)tiles,
                  it[0], it[1], it[2], bal[0], bal[1], bal[2], h->ws_bytes / 1e9, h->small_bytes / 1e6);
    s += line;
  } else {
    s += "no plan";
  }
  if (buf && len) {
    std::strncpy(buf, s.c_str(), len - 1);
    buf[len - 1] = 0;
  }
  return (int)s.size();
}

int dmuon_plan_preview(const dmuon_shape_t* shapes, int n_mats, int backend, int tile_mode, int clusters,
                       int sms, int balanced, char* buf, size_t len) {
  if (n_mats < 0 || (n_mats > 0 && !shapes) || tile_mode < 0 || tile_mode > 3 || clusters < 0 || sms < 1 ||
      (backend != DMUON_BACKEND_DIRECT && backend != DMUON_BACKEND_GRAM) ||
      (backend == DMUON_BACKEND_GRAM && clusters < 1))
    return DMUON_ERR_ARG;
  if (n_mats > 0)
    if (int rc = check_shapes(shapes, n_mats)) return rc;
  const bool gram = backend == DMUON_BACKEND_GRAM;
  std::vector<int> order;
  const int n_large = plan_order(shapes, n_mats, true, order);
  std::vector<dmuon_shape_t> ps(n_mats);
  for (int k = 0; k < n_mats; ++k) ps[k] = shapes[order[k]];
  const bool pair = choose_pairs(clusters, tile_mode, true, shapes, n_mats, gram);
  const int bn = pair ? kBN : choose_bn(sms, tile_mode, true, shapes, n_mats);
  const int procs = pair ? clusters : sms;
  size_t items[3] = {0, 0, 0}, chunks = 0;
  double busiest[3] = {0, 0, 0}, mean[3] = {0, 0, 0};
  for (const auto& cc : split_chunks(ps.data(), n_large, kDefaultChunkElems)) {
    Layout L;
    make_layout(ps.data() + cc.first, cc.second, L, pair, procs, balanced != 0, gram, bn);
    ++chunks;
    for (int q = 0; q < 3; ++q) {
      items[q] += L.items[q].size();
      const auto b = deal_balance(L, q);
      busiest[q] += b.first;
      mean[q] += b.second;
    }
  }
  char line[384];
  std::snprintf(line, sizeof line,
                "matrices %d; backend %s; tiles %s; small-matrix kernel %d; chunks %zu; "
                "items gram %zu gram2 %zu apply %zu; balance gram %.4f gram2 %.4f apply %.4f",
                n_mats, gram ? "gram" : "direct",
                pair ? "256x256 CTA pairs" : (bn == kBM ? "128x128 single CTAs" : "128x256 single CTAs"),
                n_mats - n_large, chunks, items[0], items[1], items[2],
                mean[0] > 0 ? busiest[0] / mean[0] : 1.0, mean[1] > 0 ? busiest[1] / mean[1] : 1.0,
                mean[2] > 0 ? busiest[2] / mean[2] : 1.0);
  const std::string s(line);
  if (buf && len) {
    std::strncpy(buf, s.c_str(), len - 1);
    buf[len - 1] = 0;
  }
  return (int)s.size();
}

const char* dmuon_error_string(int code) {
  switch (code) {
    case DMUON_OK: return "ok";
    case DMUON_ERR_ARG: return "invalid argument";
    case DMUON_ERR_ALIGN: return "matrix pointer not 16-byte aligned";
    case DMUON_ERR_OOM: return "out of device memory";
    case DMUON_ERR_CUDA: return "CUDA error";
    case DMUON_ERR_NONFINITE: return "non-finite input";
    case DMUON_ERR_TIMEOUT: return "kernel wait timed out";
    case DMUON_ERR_UNSUPPORTED: return "device is not compute capability 10.3 (sm_103a)";
    default: return "unknown status";
  }
}

const char* dmuon_version(void) { return kVersion; }

}  // extern "C"
