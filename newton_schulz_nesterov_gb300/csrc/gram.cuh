// Types of the Gram-space Newton-Schulz phases (ns_gram.cu).
//
// DMuon "API Reference", sections gram_newton_schulz and
// gram_newton_schulz_factors: the iteration runs on the m x m Gram matrix
// with one factor per restart window, applied to the (oriented, normalised)
// iterate.  Per step, with R = X X^T and Z = a I + b R + c R R:
//   Q <- Z Q,   R <- Z (R Z),
// and at a restart (and at the end) X <- Q X.
//
// Storage (fp16): R and W = R Z scaled by kappa, a power of two near m (at
// most 1024), which keeps their entries (~1/m unscaled) out of the fp16
// subnormal range; Z and Q unscaled, identity part included.  Z is stored
// whole rather than as a*I plus a remainder: expanding Z R Z into
// a^2 R + 2a (B R) + B (B R) cancels heavily once singular values near 1
// (Z's eigenvalue a + b + c is ~0.1..1 against a ~3..4), amplifying fp16
// rounding tenfold and more; products with Z cancel only inside the fp32
// accumulators.  The last Q of a window (buffer kGbQb) is the left operand of
// the Q X product, run by the direct Apply kernel on the fp16 iterate.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace dmuon {

// m x m buffers of one matrix, in this order in the workspace and in the
// tensor-map array.  Z alternates between Z0 and Z1 from step to step, so
// the window's first factor Q = Z is read from its Z buffer instead of being
// copied.
enum GramBuf : int {
  kGbR0 = 0, kGbR1 = 1, kGbZ0 = 2, kGbW = 3, kGbQ0 = 4, kGbQ1 = 5, kGbQb = 6, kGbZ1 = 7, kGramBufs = 8
};

// Restarts are explicit: X <- Q X (fp16, on the Apply kernel) and a new
// R <- X X^T.  (Restarting without forming X -- R <- Q R_start Q from m x m
// products, one product with X at the end -- needs fewer multiply-adds for
// n >= 2m, but keeps R_start's fp16 rounding for the whole step; an emulation
// of the roundings put it at twice the explicit restart's error and past
// 3e-2 on inputs whose singular values spread over 1e3..1e4.)

struct GramDesc {
  uint16_t* buf[kGramBufs];  // m x m fp16, leading dimension ld
  int64_t m, ld;
  float kappa, inv_kappa;    // power-of-two scale of R and W and its inverse
};

// One launch: for every item (a 256 x 256 super-tile on or above the
// diagonal of one matrix) the CTA pair computes P = opA * opB^T (both
// operands K-major; for symmetric operands that is opA * opB) and writes
//   out  = g * P + c1 * kappa^p1pow * buf[add1] + diag * I
//   out2 = the same values (another buffer; out2 >= 0)
// with g = g0 * kappa^gpow times the iterate's scale squared (xscale 1: s/p
// of X[0] = p U; 2: 1/beta' of an iterate stored as beta' X), into the tile
// and its mirror.  Operands: X[src] (fp16, K = n) for the first Gram of a
// window (x_operand = 1), else buf[opA], buf[opB] (fp16, K = m).
struct GramArgs {
  const GramDesc* gd;
  const MatDesc* mats;
  const CUtensorMap* xmaps;   // kMapsPerMat per matrix (X[0], X[1], ...)
  const CUtensorMap* gmaps;   // kGramBufs per matrix
  const int4* items;          // {mat, I, J, k_blocks}
  int n_items;
  const int* starts;          // per CTA pair: first item (see work_range), or null
  int x_operand, src;
  int opA, opB;
  int out, out2;              // out2 < 0: none
  int add1;                   // -1: none
  float g0, c1, diag;
  int gpow, p1pow, xscale;    // powers of kappa (-2..1); xscale 0 / 1 / 2 as above
  const float* svec;          // per-matrix s/p
  const float* bvec;          // per-matrix beta'
  int* err;
  unsigned long long timeout_ns;
};

cudaError_t gram_configure();
cudaError_t launch_gram_pair(const GramArgs& a, int clusters, cudaStream_t s);

}  // namespace dmuon
