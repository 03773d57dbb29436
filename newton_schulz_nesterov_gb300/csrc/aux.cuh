// Types shared by the AdamW / clipping kernels and their host launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dmuon {

// Elements per tile of the flat elementwise kernels (32 KB of fp32).
constexpr int64_t kFlatTile = 8192;

// One tensor of a flat call.  AdamW uses p, g, m, v; clipping scales g.
struct FlatDesc {
  float* p;
  const float* g;
  float* m;
  float* v;
  int64_t numel;
  int32_t bucket;   // clipping bucket
  int32_t vec4;     // 16-byte aligned pointers and numel % 4 == 0
};

struct AdamWArgs {
  const FlatDesc* descs;
  const int64_t* tile_prefix;  // n + 1
  int n;
  int64_t n_tiles;
  float decay;                 // 1 - lr*wd
  float beta1, beta2;
  float step_size;             // lr / (1 - beta1^t)
  float inv_sqrt_bc2;          // 1 / sqrt(1 - beta2^t)
  float eps;
};

struct ClipArgs {
  const FlatDesc* descs;
  const int64_t* tile_prefix;  // n + 1
  int n;
  int64_t n_tiles;
  const int* bucket_start;     // n_buckets + 1 (CSR over bucket_members)
  const int* bucket_members;   // tensor indices, bucket by bucket, in list order
  int n_buckets;
  float max_norm;              // <= 0: statistics only
  float* partials;             // n_tiles
  float* norms;                // n_buckets
  float* coefs;                // n_buckets (-1: not scaling)
};

cudaError_t launch_adamw(const AdamWArgs& a, int grid, cudaStream_t s);
cudaError_t launch_clip(const ClipArgs& a, int grid, cudaStream_t s);

}  // namespace dmuon
