// Types of the fused small-matrix Muon step (ns_small.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dmuon {

// Oriented shapes handled by the fused kernel: m <= 128, n <= 512.
constexpr int kSmallMaxM = 128;
constexpr int kSmallMaxN = 512;
constexpr int kSmallBlockBytes = 128 * 128;  // one 64-column block of 128 rows (fp16)
constexpr int kSmallThreads = 256;
constexpr int kSmallSmem = 1024 /*align slack*/ + 12 * kSmallBlockBytes + 256;

struct SmallDesc {
  int64_t rows, cols;   // weight shape
  int32_t idx;          // position in the pointer list (and flag index)
  float scale;          // update scale of this matrix
};

struct SmallArgs {
  const SmallDesc* descs;   // one per CTA
  const MatPtrs* ptrs;
  int* flags;
  int* err;
  unsigned long long timeout_ns;  // product wait limit (0: 4 s)
  int ns_steps;
  int ns_only;
  int nesterov;
  float mu, eps, lr, decay;
  float coeffs[64][3];      // per-iteration (a, b, c)
};

cudaError_t small_configure();
cudaError_t launch_small(const SmallArgs& a, int n_mats, cudaStream_t s);

}  // namespace dmuon
