// Shared device-side types and PTX helpers of the GB300 Muon step.
//
// Plan-time descriptors (one per matrix), per-call pointers, the work-item
// encoding of the tensor-core phases and thin inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (MMA, TMEM).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dmuon {

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------

// One matrix of the packed list, oriented so that the Newton-Schulz iterate
// X is m x n with m <= n (m = short side).  X, A and B live in the handle's
// workspace; W, G, M are the caller's (see MatPtrs).
//
// The iterate and the products are fp16 with power-of-two scales that keep
// their entries inside fp16's normal range (fp16 has three more mantissa
// bits than bf16; power-of-two scaling is exact):
//   X[0] holds p U (oriented, p a per-matrix power of two chosen by the
//        momentum pass so that max |p U| lies in [2^6, 2^14]);
//   X[k] (after the first product) holds beta' X with beta' = beta / nu
//        (beta ~ sqrt(n), a power of two; nu = ||X0||_F rounded down to a
//        power of two when below 1/2, else 1 -- X0 = U / (||U|| + eps) has
//        a norm far below 1 when ||U|| is far below eps), so the iterate's
//        entries stay near 1 whatever the input's scale;
//   A holds kappa X X^T, kappa ~ m (at most 1024);
//   B holds Z = a I + b A + c A A (unscaled; its entries are O(a)).
struct MatDesc {
  int64_t rows, cols;      // weight shape (row-major fp32)
  int64_t m, n;            // oriented iterate shape, m = min(rows, cols)
  int64_t ldx;             // leading dimension (elements) of X buffers
  int64_t lda;             // leading dimension (elements) of A and B
  __half* X[2];            // ping/pong iterate, m x n row-major
  __half* A;               // kappa X X^T, m x m
  __half* B;               // Z (or b*A + c*A*A), m x m
  int64_t tile0;           // first momentum tile of this matrix
  int32_t tiles_c;         // momentum tiles along cols
  int32_t transposed;      // rows > cols
  float scale;             // update scale of this matrix
  float kappa;             // scale of A: largest power of two <= min(m, 1024)
  float beta;              // power of two nearest sqrt(n) (times 1/nu per call: bvec)
  int32_t sym_items;       // work items of this matrix in each symmetric phase (Gram, Gram2)
  int32_t apply_items;     // work items of this matrix in each Apply phase
  int32_t pad_;
};

// Power-of-two scales of a matrix's fp16 buffers (host and device).
__host__ __device__ inline float scale_kappa(int64_t m) {
  float k = 1.f;
  while (k * 2.f <= (float)(m < 1024 ? m : 1024)) k *= 2.f;
  return k;
}
__host__ __device__ inline float scale_beta(int64_t n) {
  // 2^round(log2(sqrt(n))): the largest power of two whose square is at most 2n
  float b = 1.f;
  while ((double)(2.f * b) * (double)(2.f * b) <= 2.0 * (double)n) b *= 2.f;
  return b;
}

// Caller pointers of one call (uploaded only when they change).
struct MatPtrs {
  float* W;        // parameters (dmuon_step) or output O (newton_schulz)
  const float* G;  // gradient / NS input
  float* M;        // momentum buffer (unused by newton_schulz)
  void* pad_;
};

// Momentum/normalisation tile: 64 x 64 fp32 elements of W's shape.
constexpr int kMomTile = 64;

// Work item of a tensor-core phase: {matrix, row tile, 256-col tile, number
// of 64-wide K blocks}; the row tile is 128 rows for single CTAs and 256 rows
// for CTA pairs.
// Single-CTA tile: 128 rows (UMMA M) x 256 cols (UMMA N), K step 64.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kBox = 64;                        // TMA box is 64 x 64 16-bit values
constexpr int kBoxBytes = kBox * kBox * 2;      // 8 KB
constexpr int kGemmThreads = 192;               // TMA, MMA, 4 epilogue warps
constexpr int kTmemCols = 512;                  // two 128x256 fp32 accumulators
constexpr int kEpiWords = 32 * 17;              // per-warp transpose scratch
constexpr int kGemmSmem =
    1024 /*align slack*/ + kStages * kStageBytes + 4 * kEpiWords * 4 + 256;

// CTA-pair variant (cta_group::2): a 2-CTA cluster computes a 256x256 tile,
// each CTA loading its 128 rows of A and its 128-row half of B per K block,
// so a stage is 32 KB per CTA and six stages fit.
constexpr int kPairStages = 6;
constexpr int kPairHalfBytes = 128 * kBK * 2;            // 16 KB
constexpr int kPairStageBytes = 2 * kPairHalfBytes;      // 32 KB per CTA
constexpr int kPairSmem =
    1024 /*align slack*/ + kPairStages * kPairStageBytes + 4 * kEpiWords * 4 + 256;

enum Phase : int { kPhaseGram = 0, kPhaseGram2 = 1, kPhaseApply = 2, kPhaseFused = 3 };
enum FinalMode : int { kWriteX = 0, kUpdateW = 1, kWriteO = 2 };

// Tensor maps per matrix: X[0], X[1], A, B (box 64x64, 128B swizzle).
constexpr int kMapsPerMat = 4;

struct GemmArgs {
  const MatDesc* mats;
  const MatPtrs* ptrs;
  const CUtensorMap* tmaps;
  const int4* items;       // {mat, ti, tj, k_blocks}
  int n_items;
  const int* starts;       // balanced dealing: processor c runs items [starts[c], starts[c+1]); null: c, c+P, ...
  int src;                 // X buffer holding the current iterate
  float ca, cb, cc;        // this iteration's (a, b, c)
  int first;               // first iteration: fold the norm scale in
  int fold;                // Gram2 adds a*I (B becomes Z = aI + B); Apply then skips its a*X term
  int final_mode;          // Apply phase: kWriteX / kUpdateW / kWriteO
  float lr, decay;         // W <- decay*W - lr*scale*O
  const float* svec;       // per-matrix s/p: X[0] times this is U / (||U||_F + eps)
  const float* bvec;       // per-matrix beta': X[k] (k >= 1) holds beta' X
  int* err;                // device error word (bit 0: wait timeout)
  unsigned long long timeout_ns;  // wait without progress before giving up (0 = 4 s)
  // Fused launches (kPhaseFused): every stage s = 3k + p (iteration k, phase
  // p) of every matrix in one launch.  Each processor runs, for k = 0 ..
  // n_iters-1 and p = 0, 1, 2, its share of phase p's dealt list (fitems[p],
  // fstarts[p] over fprocs[p] processors; the lists of the per-phase
  // launches); a tile of stage s waits until its matrix's counter shows every
  // tile of the stages before s done (each epilogue warp adds 1 per finished
  // tile).  coef[k] is iteration k's (a, b, c); the last iteration's Apply
  // uses final_mode, earlier ones write X.
  const int4* fitems[3];
  const int* fstarts[3];
  int fn_items[3];
  int fprocs[3];
  int n_iters;
  int* counters;           // per matrix, zero at launch
  float coef[64][3];
  // Operand precision: iteration k multiplies fp16 operands when k <
  // f16_iters, else bf16 (same scales).  Per-phase launches give their
  // iteration in `iter`; X0 is always fp16 (f16_iters >= 1).
  int iter;
  int f16_iters;
};

// Items of one persistent processor (a CTA, or a CTA pair): its own run
// [starts[proc], starts[proc + 1]) when the host dealt the list (the launch
// then has exactly as many processors as starts has entries minus one), else
// every nproc-th item from proc on.
struct WorkRange { int w0, w1, step; };
__device__ __forceinline__ WorkRange work_range(const int* starts, int proc, int nproc, int n_items) {
  if (starts) return WorkRange{starts[proc], starts[proc + 1], 1};
  return WorkRange{proc, n_items, nproc};
}

// Momentum pass.  X[0] = fp16(p U) with p = pscale[matrix], a power of two
// kept from the previous step (the norm is only known after the pass).  The
// finalisation checks max |U| * p against [2^6, 2^14] -- no fp16 overflow,
// no precision lost to subnormals -- and, when it misses, picks a new p and
// flags the matrix; the redo pass (redo = 1) then rewrites X[0] and the tile
// sums of the flagged matrices from G and the updated M (the same U, bit for
// bit) and a second finalisation completes them.
// Resident CTAs per SM of the momentum kernel (its launch bound); a launch
// needs no more than num_sms * kMomCtasPerSm CTAs (they stride over tiles).
constexpr int kMomCtasPerSm = 4;

struct MomArgs {
  const MatDesc* mats;
  const MatPtrs* ptrs;
  const int64_t* tile_prefix;  // n_mats + 1 entries
  int n_mats;
  int64_t n_tiles;
  float mu;
  int nesterov;
  int ns_only;                 // 1: U = G (standalone NS), no momentum
  float* partials;             // per-tile sum of squares of p U
  float* tmax;                 // per-tile max |U| (written by the first pass only)
  const float* pscale;         // per-matrix prescale p
  const int* redo;             // per-matrix redo flags (redo pass)
  int redo_pass;               // 0: momentum pass; 1: rewrite flagged matrices only
};

struct FinalizeArgs {
  const MatDesc* mats;
  const int64_t* tile_prefix;
  const float* partials;
  const float* tmax;
  int n_mats;
  float eps;
  float* svec;                 // s / p
  float* bvec;                 // beta' = beta / nu, the scale of X after the first product
  float* pscale;               // p, replaced when it misses its window
  int* redo;                   // per-matrix: 1 = X[0] must be rewritten with the new p
  int* flags;
  int redo_pass;               // 1: finish the flagged matrices only, clearing their flag
};

struct Update0Args {          // ns_steps == 0: O = (s/p) X[0] straight to W / out
  const MatDesc* mats;
  const MatPtrs* ptrs;
  const int64_t* tile_prefix;
  int n_mats;
  int64_t n_tiles;
  const float* svec;
  float lr, decay;
  int write_o;
};

// Host launchers (defined in the .cu files).
cudaError_t launch_mom(const MomArgs& a, int grid, cudaStream_t s);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s);
cudaError_t launch_update0(const Update0Args& a, int grid, cudaStream_t s);
// Single-CTA launches; bn: tile width (256, or 128 for narrow plans).
cudaError_t launch_gemm(int phase, const GemmArgs& a, int grid, cudaStream_t s, int bn = kBN);
cudaError_t gemm_configure();
// CTA-pair kernels: items are {matrix, 256-row tile, 256-col tile, K blocks};
// `clusters` 2-CTA clusters are launched.
cudaError_t launch_gemm_pair(int phase, const GemmArgs& a, int clusters, cudaStream_t s);
cudaError_t gemm_pair_configure(int* max_clusters);

}  // namespace dmuon
