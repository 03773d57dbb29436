// HBM-bound kernels of the Muon step: fused momentum / Nesterov / orientation
// / sum-of-squares writing the fp16 iterate, the per-matrix norm finalisation
// (with the redo pass for a prescale that missed), and the ns_steps == 0
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

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One CTA iteration handles a 64x64 tile of W's shape.  256 threads: thread
// t covers columns 4*(t%16)..+3 of rows t/16 + 16*i, i = 0..3, so each warp
// reads two full 256-byte row segments per array (coalesced float4).
// Momentum pass (redo_pass = 0):
//   M <- mu*M + G ;  U = G + mu*M (nesterov) or M ;  X0 <- fp16(p U or p U^T)
//   partials[tile] = sum((p U)^2), tmax[tile] = max |U|, fixed reduction order.
// Redo pass (REDO): only tiles of matrices flagged by the finalisation; U is
// recomputed from G and the already updated M (the same fmaf sequence, so the
// same U) and X0 and partials are rewritten with the matrix's new p.  A CTA
// that finds no flagged matrix returns at once.
// Up to 64 registers a thread (kMomCtasPerSm CTAs per SM), so that the eight
// 16-byte loads of a tile's four rows are all in flight before its stores.
template <bool REDO>
__global__ void __launch_bounds__(256, kMomCtasPerSm) mom_norm_kernel(const MomArgs a) {
  __shared__ uint32_t stage[kMomTile * 33];  // 64 x 66 fp16, odd word stride
  __shared__ float red[8];
  __shared__ float redm[8];
  __shared__ int any;
  __half* st = reinterpret_cast<__half*>(stage);
  const int tid = threadIdx.x;
  const int cl = (tid & 15) * 4;
  const int rl0 = tid >> 4;
  constexpr bool redo_pass = REDO;

  if (redo_pass) {
    if (tid == 0) any = 0;
    __syncthreads();
    int mine = 0;
    for (int i = tid; i < a.n_mats; i += blockDim.x) mine |= a.redo[i];
    if (mine) any = 1;
    __syncthreads();
    if (!any) return;
  }

  int mi = 0;
  int64_t mt0 = 0, mt1 = 0;  // tiles of matrix mi: the search is skipped while t stays inside
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    if (t < mt0 || t >= mt1) {
      mi = find_mat(a.tile_prefix, a.n_mats, t);
      mt0 = __ldg(a.tile_prefix + mi);
      mt1 = __ldg(a.tile_prefix + mi + 1);
    }
    if (redo_pass && !a.redo[mi]) continue;  // uniform over the CTA
    const MatDesc& d = a.mats[mi];
    const MatPtrs& p = a.ptrs[mi];
    const float ps = a.pscale[mi];
    const int64_t rows = d.rows, cols = d.cols;
    const int64_t local = t - d.tile0;
    const int64_t r0 = (local / d.tiles_c) * kMomTile;
    const int64_t c0 = (local % d.tiles_c) * kMomTile;
    const int64_t c = c0 + cl;
    const bool vec = (cols & 3) == 0;
    const bool tr = d.transposed != 0;
    __half* X = d.X[0];
    const int64_t ldx = d.ldx;
    float ss = 0.f, mx = 0.f;

    // Every load of the tile's four rows is issued before any store: the
    // compiler may not move a load above a store to memory it might alias.
    float4 gv[4], mv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = r0 + rl0 + 16 * i;
      if (vec && r < rows && c < cols) {
        gv[i] = ld_once(p.G + r * cols + c);
        if (!a.ns_only) mv[i] = ld_once(p.M + r * cols + c);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rl = rl0 + 16 * i;
      const int64_t r = r0 + rl;
      float u[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < rows && c < cols) {
        const int64_t off = r * cols + c;
        if (vec) {
          const float4 g4 = gv[i];
          const float g[4] = {g4.x, g4.y, g4.z, g4.w};
          if (a.ns_only) {
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = g[j];
          } else if (redo_pass) {
            const float4 m4 = mv[i];  // already mu*M + G
            const float mn[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = a.nesterov ? fmaf(a.mu, mn[j], g[j]) : mn[j];
          } else {
            const float4 m4 = mv[i];
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
              } else if (redo_pass) {
                const float mn = p.M[off + j];
                u[j] = a.nesterov ? fmaf(a.mu, mn, g) : mn;
              } else {
                const float mn = fmaf(a.mu, p.M[off + j], g);
                p.M[off + j] = mn;
                u[j] = a.nesterov ? fmaf(a.mu, mn, g) : mn;
              }
            }
          }
        }
      }
      float x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[j] = u[j] * ps;  // a power of two: exact unless out of fp32 range
        ss = fmaf(x[j], x[j], ss);
        mx = fmaxf(mx, fabsf(u[j]));
      }

      if (!tr) {
        if (r < rows && c < cols) {
          __half* dst = X + r * ldx + c;
          if (c + 4 <= cols) {
            uint2 v;
            v.x = pack_h2(x[0], x[1]);
            v.y = pack_h2(x[2], x[3]);
            *reinterpret_cast<uint2*>(dst) = v;
          } else {
            for (int j = 0; j < 4 && c + j < cols; ++j) dst[j] = __float2half_rn(x[j]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) st[(cl + j) * 66 + rl] = __float2half_rn(x[j]);
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
          __half* dst = X + xr * ldx + xc;
          if (xc + 8 <= d.n) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            for (int j = 0; j < 8 && xc + j < d.n; ++j) dst[j] = st[cr * 66 + seg + j];
          }
        }
      }
    }

    // Deterministic tile sum: fixed shuffle tree, then warps in order (the
    // maximum does not depend on the order).
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((tid & 31) == 0) {
      red[tid >> 5] = ss;
      redm[tid >> 5] = mx;
    }
    __syncthreads();
    if (tid == 0) {
      float s = 0.f, m = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        s += red[w];
        m = fmaxf(m, redm[w]);
      }
      a.partials[t] = s;
      if (!redo_pass) a.tmax[t] = m;
    }
    __syncthreads();
  }
}

// s/p and beta' of a matrix from S = sum (p U)^2: X0 * (s/p) = U / (||U|| + eps)
// with ||U|| = sqrt(S) / p, and nu = ||X0||_F = sqrt(S) / (sqrt(S) + eps p);
// beta' = beta / 2^floor(log2 nu) when nu < 1/2 (at most 2^100), else beta.
__device__ __forceinline__ void set_scales(const FinalizeArgs& a, int mi, double tot, double p, float beta) {
  const double r = sqrt(tot), den = r + (double)a.eps * p;
  a.svec[mi] = (float)(1.0 / den);
  const double nu = r / den;
  float b = beta;
  if (nu < 0.5 && nu > 0.0) {
    int ex = 0;
    frexp(nu, &ex);  // nu = f 2^ex, f in [0.5, 1): floor(log2 nu) = ex - 1
    b = ldexpf(beta, min(100, 1 - ex));
  }
  a.bvec[mi] = b;
}

// One CTA per matrix: fp64 sum of the tile partials in a fixed order (the
// sum of (p U)^2) and the maximum of |U|.  Then, with S the sum:
//   non-finite input (S NaN or max |U| infinite): flag, s/p = 0;
//   zero input: s/p = 0 (X0 = 0, so every output is 0);
//   max |U| * p inside [2^6, 2^14] and S finite: s/p and beta' (set_scales);
//   otherwise: p <- 2^(11 - e) with max |U| = f 2^e, f in [0.5, 1) (so that
//     max |p U| lies in [2^10, 2^11)), and the matrix is flagged for the redo
//     pass, whose second finalisation (redo_pass = 1) computes s/p from the
//     rewritten partials and clears the flag.
__global__ void __launch_bounds__(256) finalize_kernel(const FinalizeArgs a) {
  __shared__ double red[256];
  __shared__ float redm[256];
  const int mi = blockIdx.x;
  if (a.redo_pass && !a.redo[mi]) return;
  const int64_t b = a.tile_prefix[mi], e = a.tile_prefix[mi + 1];
  double s = 0.0;
  float mx = 0.f;
  for (int64_t i = b + threadIdx.x; i < e; i += blockDim.x) {
    s += (double)a.partials[i];
    if (!a.redo_pass) mx = fmaxf(mx, a.tmax[i]);
  }
  red[threadIdx.x] = s;
  redm[threadIdx.x] = mx;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) {
      red[threadIdx.x] += red[threadIdx.x + w];
      redm[threadIdx.x] = fmaxf(redm[threadIdx.x], redm[threadIdx.x + w]);
    }
    __syncthreads();
  }
  if (threadIdx.x != 0) return;
  const double tot = red[0];
  const double p = (double)a.pscale[mi];
  const float beta = a.mats[mi].beta;
  if (a.redo_pass) {
    set_scales(a, mi, tot, p, beta);
    a.redo[mi] = 0;
    return;
  }
  const float m = redm[0];
  if (isnan(tot) || isinf(m)) {
    a.svec[mi] = 0.f;
    a.bvec[mi] = beta;
    a.flags[mi] |= 1;
    return;
  }
  if (m == 0.f) {
    a.svec[mi] = 0.f;
    a.bvec[mi] = beta;
    return;
  }
  const double q = (double)m * p;
  if (isfinite(tot) && q >= 64.0 && q <= 16384.0) {
    set_scales(a, mi, tot, p, beta);
    return;
  }
  int ex = 0;
  frexpf(m, &ex);
  const int k = min(127, max(-126, 11 - ex));
  a.pscale[mi] = ldexpf(1.f, k);
  a.redo[mi] = 1;
}

// ns_steps == 0: O = (s/p) * X0 (oriented back), then the update or a plain
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
      const float o = s * __half2float(d.X[0][xoff]);
      float* w = p.W + r * d.cols + c;
      *w = a.write_o ? o : fmaf(a.decay, *w, -coef * o);
    }
  }
}

}  // namespace

cudaError_t launch_mom(const MomArgs& a, int grid, cudaStream_t s) {
  if (a.redo_pass)
    mom_norm_kernel<true><<<grid, 256, 0, s>>>(a);
  else
    mom_norm_kernel<false><<<grid, 256, 0, s>>>(a);
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
