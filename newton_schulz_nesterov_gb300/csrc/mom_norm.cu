// HBM-bound kernels of the Muon step: fused momentum / Nesterov / orientation
// / sum-of-squares, the per-matrix norm finalisation, and the ns_steps == 0
// update.
//
// DMuon "API Reference", section "Muon": momentum buffer update and the
// Nesterov input (gradient + momentum * buffer, buffer taken after this
// step's update).  Section "gram_newton_schulz_factors": the normaliser is
// the Frobenius norm plus eps of the (possibly transposed) input.
#include "common.cuh"

namespace dmuon {

namespace {

__device__ __forceinline__ int find_mat(const int64_t* prefix, int n, int64_t t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(prefix + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float4 ld_once(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));  // streamed: read once
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One CTA iteration handles a 64x64 tile of W's shape.  256 threads: thread
// t covers columns 4*(t%16)..+3 of rows t/16 + 16*i, i = 0..3, so each warp
// reads two full 256-byte row segments per array (coalesced float4).
//   M <- mu*M + G ;  U = G + mu*M (nesterov) or M ;  X0 <- bf16(U or U^T)
//   partials[tile] = sum(U^2) over the tile, fixed reduction order.
__global__ void __launch_bounds__(256) mom_norm_kernel(const MomArgs a) {
  __shared__ uint32_t stage[kMomTile * 33];  // 64 x 66 bf16, odd word stride
  __shared__ float red[8];
  __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stage);
  const int tid = threadIdx.x;
  const int cl = (tid & 15) * 4;
  const int rl0 = tid >> 4;

  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const int mi = find_mat(a.tile_prefix, a.n_mats, t);
    const MatDesc& d = a.mats[mi];
    const MatPtrs& p = a.ptrs[mi];
    const int64_t rows = d.rows, cols = d.cols;
    const int64_t local = t - d.tile0;
    const int64_t r0 = (local / d.tiles_c) * kMomTile;
    const int64_t c0 = (local % d.tiles_c) * kMomTile;
    const int64_t c = c0 + cl;
    const bool vec = (cols & 3) == 0;
    const bool tr = d.transposed != 0;
    __nv_bfloat16* X = d.X[0];
    const int64_t ldx = d.ldx;
    float ss = 0.f;

#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rl = rl0 + 16 * i;
      const int64_t r = r0 + rl;
      float u[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < rows && c < cols) {
        const int64_t off = r * cols + c;
        if (vec) {
          const float4 g4 = ld_once(p.G + off);
          const float g[4] = {g4.x, g4.y, g4.z, g4.w};
          if (a.ns_only) {
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = g[j];
          } else {
            const float4 m4 = ld_once(p.M + off);
            const float mo[4] = {m4.x, m4.y, m4.z, m4.w};
            float mn[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              mn[j] = fmaf(a.mu, mo[j], g[j]);
              u[j] = a.nesterov ? fmaf(a.mu, mn[j], g[j]) : mn[j];
            }
            __stcs(reinterpret_cast<float4*>(p.M + off),
                   make_float4(mn[0], mn[1], mn[2], mn[3]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (c + j < cols) {
              const float g = p.G[off + j];
              if (a.ns_only) {
                u[j] = g;
              } else {
                const float mn = fmaf(a.mu, p.M[off + j], g);
                p.M[off + j] = mn;
                u[j] = a.nesterov ? fmaf(a.mu, mn, g) : mn;
              }
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(u[j], u[j], ss);

      if (!tr) {
        if (r < rows && c < cols) {
          __nv_bfloat16* dst = X + r * ldx + c;
          if (c + 4 <= cols) {
            uint2 v;
            v.x = pack_bf16x2(u[0], u[1]);
            v.y = pack_bf16x2(u[2], u[3]);
            *reinterpret_cast<uint2*>(dst) = v;
          } else {
            for (int j = 0; j < 4 && c + j < cols; ++j) dst[j] = __float2bfloat16_rn(u[j]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) st[(cl + j) * 66 + rl] = __float2bfloat16_rn(u[j]);
      }
    }

    if (tr) {
      // X = U^T: X row = W column, X column = W row.  8 threads per X row,
      // 16 bytes each, two passes of 32 rows.
      __syncthreads();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const int cr = (tid >> 3) + 32 * pass;
        const int seg = (tid & 7) * 8;
        const int64_t xr = c0 + cr;
        const int64_t xc = r0 + seg;
        if (xr < d.m && xc < d.n) {
          const uint32_t* w = stage + cr * 33 + seg / 2;
          __nv_bfloat16* dst = X + xr * ldx + xc;
          if (xc + 8 <= d.n) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            for (int j = 0; j < 8 && xc + j < d.n; ++j) dst[j] = st[cr * 66 + seg + j];
          }
        }
      }
    }

    // Deterministic tile sum: fixed shuffle tree, then warps in order.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) s += red[w];
      a.partials[t] = s;
    }
    __syncthreads();
  }
}

// One CTA per matrix: fp64 sum of the tile partials in a fixed order, then
// s = 1 / (sqrt(sum) + eps).  A non-finite sum sets the matrix's flag.
__global__ void __launch_bounds__(256) finalize_kernel(const FinalizeArgs a) {
  __shared__ double red[256];
  const int mi = blockIdx.x;
  const int64_t b = a.tile_prefix[mi], e = a.tile_prefix[mi + 1];
  double s = 0.0;
  for (int64_t i = b + threadIdx.x; i < e; i += blockDim.x) s += (double)a.partials[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tot = red[0];
    const bool finite = isfinite(tot);
    const double nrm = sqrt(tot) + (double)a.eps;
    a.svec[mi] = finite ? (float)(1.0 / nrm) : 0.f;
    if (!finite) a.flags[mi] |= 1;
  }
}

// ns_steps == 0: O = s * X0 (oriented back), then the update or a plain
// write of O.  Scalar, one element per thread iteration; only used for this
// degenerate step count.
__global__ void __launch_bounds__(256) update0_kernel(const Update0Args a) {
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const int mi = find_mat(a.tile_prefix, a.n_mats, t);
    const MatDesc& d = a.mats[mi];
    const MatPtrs& p = a.ptrs[mi];
    const int64_t local = t - d.tile0;
    const int64_t r0 = (local / d.tiles_c) * kMomTile;
    const int64_t c0 = (local % d.tiles_c) * kMomTile;
    const float s = a.svec[mi];
    const float coef = a.lr * d.scale;
    for (int e = threadIdx.x; e < kMomTile * kMomTile; e += blockDim.x) {
      const int64_t r = r0 + e / kMomTile, c = c0 + e % kMomTile;
      if (r >= d.rows || c >= d.cols) continue;
      const int64_t xoff = d.transposed ? c * d.ldx + r : r * d.ldx + c;
      const float o = s * __bfloat162float(d.X[0][xoff]);
      float* w = p.W + r * d.cols + c;
      *w = a.write_o ? o : fmaf(a.decay, *w, -coef * o);
    }
  }
}

}  // namespace

cudaError_t launch_mom(const MomArgs& a, int grid, cudaStream_t s) {
  mom_norm_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s) {
  finalize_kernel<<<a.n_mats, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_update0(const Update0Args& a, int grid, cudaStream_t s) {
  update0_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dmuon
