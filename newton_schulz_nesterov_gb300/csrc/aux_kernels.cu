// HBM-bound kernels for the rest of Muon.step: AdamW on the non-Muon
// parameters and segmented gradient-norm clipping.
//
// DMuon "API Reference", section "Muon": symmetric (non-dedicated) parameters
// take AdamW (defaults lr 1e-3, betas (0.9, 0.999), weight decay 0.01,
// eps 1e-8); sections "clip_grad_norm_" and "clip_grad_norm_buckets_": each
// bucket of gradients has its own norm and clip coefficient.
//
// Both work on flat tensor lists cut into tiles of kFlatTile elements; a
// grid-stride loop over the tile list finds each tile's tensor by binary
// search of the tile prefix sums.  Full float4 accesses when the tensor is
// 16-byte aligned and its length a multiple of 4, scalar ones otherwise.
#include "aux.cuh"

namespace dmuon {

namespace {

__device__ __forceinline__ int find_tensor(const int64_t* prefix, int n, int64_t t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(prefix + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One AdamW element, in the order PyTorch's AdamW uses:
//   p *= 1 - lr*wd; m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
//   p -= (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps)
struct AdamWScalars {
  float decay, b1, b2, omb1, omb2, step_size, inv_sqrt_bc2, eps;
};

__device__ __forceinline__ void adamw_elem(const AdamWScalars& s, float& p, float g, float& m, float& v) {
  p *= s.decay;
  m = fmaf(s.b1, m, s.omb1 * g);
  v = fmaf(s.b2, v, s.omb2 * g * g);
  const float denom = sqrtf(v) * s.inv_sqrt_bc2 + s.eps;
  p = fmaf(-s.step_size, m / denom, p);
}

__global__ void __launch_bounds__(256) adamw_kernel(const AdamWArgs a) {
  const AdamWScalars s{a.decay, a.beta1, a.beta2, 1.f - a.beta1, 1.f - a.beta2, a.step_size,
                       a.inv_sqrt_bc2, a.eps};
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const int ti = find_tensor(a.tile_prefix, a.n, t);
    const FlatDesc& d = a.descs[ti];
    const int64_t base = (t - a.tile_prefix[ti]) * kFlatTile;
    const int64_t len = min((int64_t)kFlatTile, d.numel - base);
    if (d.vec4) {
      float4* p4 = reinterpret_cast<float4*>(d.p + base);
      const float4* g4 = reinterpret_cast<const float4*>(d.g + base);
      float4* m4 = reinterpret_cast<float4*>(d.m + base);
      float4* v4 = reinterpret_cast<float4*>(d.v + base);
      for (int64_t i = threadIdx.x; i < len / 4; i += blockDim.x) {
        float4 p = __ldcs(p4 + i), m = __ldcs(m4 + i), v = __ldcs(v4 + i);
        const float4 g = __ldcs(g4 + i);
        adamw_elem(s, p.x, g.x, m.x, v.x);
        adamw_elem(s, p.y, g.y, m.y, v.y);
        adamw_elem(s, p.z, g.z, m.z, v.z);
        adamw_elem(s, p.w, g.w, m.w, v.w);
        __stcs(p4 + i, p);
        __stcs(m4 + i, m);
        __stcs(v4 + i, v);
      }
    } else {
      for (int64_t i = threadIdx.x; i < len; i += blockDim.x) {
        float p = d.p[base + i], m = d.m[base + i], v = d.v[base + i];
        adamw_elem(s, p, d.g[base + i], m, v);
        d.p[base + i] = p;
        d.m[base + i] = m;
        d.v[base + i] = v;
      }
    }
  }
}

// Per-tile sum of squares in a fixed order: each thread runs over a fixed
// subset (elements threadIdx.x, +256, +512, ... of the tile, in that order),
// then a shuffle tree and the warps in order.  Four CTAs per SM with up to 64
// registers a thread, so that a whole tile's loads (eight 16-byte reads per
// thread) are in flight before any is summed.
constexpr int kSumsqCtasPerSm = 4;
__global__ void __launch_bounds__(256, kSumsqCtasPerSm) sumsq_kernel(const ClipArgs a) {
  __shared__ float red[8];
  int ti = 0;
  int64_t t0 = 0, t1 = 0;  // tiles of tensor ti: the search is skipped while t stays inside
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    if (t < t0 || t >= t1) {
      ti = find_tensor(a.tile_prefix, a.n, t);
      t0 = __ldg(a.tile_prefix + ti);
      t1 = __ldg(a.tile_prefix + ti + 1);
    }
    const FlatDesc& d = a.descs[ti];
    const int64_t base = (t - t0) * kFlatTile;
    const int64_t len = min((int64_t)kFlatTile, d.numel - base);
    float ss = 0.f;
    if (d.vec4) {
      // A full tile is 2048 float4 over 256 threads: 8 per thread.
      constexpr int kPer = kFlatTile / 4 / 256;
      const float4* g4 = reinterpret_cast<const float4*>(d.g + base);
      const int64_t nv = len / 4;
      float4 q[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int64_t i = threadIdx.x + (int64_t)k * 256;
        q[k] = i < nv ? __ldcs(g4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        ss = fmaf(q[k].x, q[k].x, ss);
        ss = fmaf(q[k].y, q[k].y, ss);
        ss = fmaf(q[k].z, q[k].z, ss);
        ss = fmaf(q[k].w, q[k].w, ss);
      }
    } else {
      for (int64_t i = threadIdx.x; i < len; i += blockDim.x) {
        const float g = d.g[base + i];
        ss = fmaf(g, g, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < 8; ++w) s += red[w];
      a.partials[t] = s;
    }
    __syncthreads();
  }
}

// One block per bucket: fp64 sum over the bucket's tensors (in list order)
// and their tiles, fixed order; then norm and clip coefficient.
__global__ void __launch_bounds__(256) clip_finalize_kernel(const ClipArgs a) {
  __shared__ double red[256];
  const int b = blockIdx.x;
  double s = 0.0;
  for (int k = a.bucket_start[b]; k < a.bucket_start[b + 1]; ++k) {
    const int ti = a.bucket_members[k];
    for (int64_t t = a.tile_prefix[ti] + threadIdx.x; t < a.tile_prefix[ti + 1]; t += blockDim.x)
      s += (double)a.partials[t];
  }
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double nrm = sqrt(red[0]);
    a.norms[b] = (float)nrm;
    // A negative coefficient means "statistics only, do not scale".
    a.coefs[b] = a.max_norm > 0.f ? (float)((double)a.max_norm / (nrm + 1e-6)) : -1.f;
  }
}

__global__ void __launch_bounds__(256) clip_scale_kernel(const ClipArgs a) {
  int ti = 0;
  int64_t t0 = 0, t1 = 0;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    if (t < t0 || t >= t1) {
      ti = find_tensor(a.tile_prefix, a.n, t);
      t0 = __ldg(a.tile_prefix + ti);
      t1 = __ldg(a.tile_prefix + ti + 1);
    }
    const FlatDesc& d = a.descs[ti];
    const float c = a.coefs[d.bucket];
    if (!(c >= 0.f && c < 1.f)) continue;  // no clipping for this bucket (NaN too)
    const int64_t base = (t - t0) * kFlatTile;
    const int64_t len = min((int64_t)kFlatTile, d.numel - base);
    float* g = const_cast<float*>(d.g) + base;
    if (d.vec4) {
      float4* g4 = reinterpret_cast<float4*>(g);
      for (int64_t i = threadIdx.x; i < len / 4; i += blockDim.x) {
        float4 x = __ldcs(g4 + i);
        x.x *= c; x.y *= c; x.z *= c; x.w *= c;
        __stcs(g4 + i, x);
      }
    } else {
      for (int64_t i = threadIdx.x; i < len; i += blockDim.x) g[i] *= c;
    }
  }
}

}  // namespace

cudaError_t launch_adamw(const AdamWArgs& a, int grid, cudaStream_t s) {
  adamw_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_clip(const ClipArgs& a, int grid, cudaStream_t s) {
  // grid: up to eight CTAs per SM; the sum of squares keeps half of them
  // resident (its launch bound) and strides over the tiles.
  sumsq_kernel<<<(grid + 1) / 2, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  clip_finalize_kernel<<<a.n_buckets, 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.max_norm > 0.f) {
    clip_scale_kernel<<<grid, 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace dmuon
