// Fused Muon step for small matrices: one CTA runs a matrix's whole step
// -- momentum, Nesterov input, norm, ns_steps quintic Newton-Schulz
// iterations and the update -- with the iterate, A and B resident in shared
// memory and the products accumulated in TMEM.  For oriented shapes with
// m <= 128 and n <= 512 (DMuon "Quick Start": TinyMLP projections at small
// widths; 64x256 tensor-parallel shards): X is at most 128 x 512 bf16 =
// 128 KB, A and B 32 KB each.
//
// DMuon "API Reference", section "direct_newton_schulz": per step
//   A = X X^T,  B = b A + c A A,  X = a X + B X;
// section "Muon": momentum and the Nesterov input; section
// "gram_newton_schulz_factors": normaliser = Frobenius norm + eps under the
// orientation rule.
//
// Shared-memory layout: each matrix is stored as 64-column blocks of
// 128 rows x 128 bytes with the 128-byte swizzle (16-byte chunk index XOR
// row % 8), the layout TMA writes for 64x128 boxes.  The same X layout is the
// K-major operand of X X^T (rows of X, K along columns) and the MN-major B
// operand of B X (K along rows, N along columns); A and B are K-major.
//
// 128 threads: thread i owns row i (TMEM lane i) in every epilogue; thread 0
// issues the MMAs (M = 128, fp32 accumulate, bf16 operands).  Every product
// completes on one mbarrier with a bounded wait.
#include "common.cuh"
#include "ptx.cuh"
#include "small.cuh"

namespace dmuon {

namespace {

constexpr uint64_t kSmallTimeoutNs = 4000000000ull;  // default product wait limit
constexpr uint64_t kSmallDrainNs = 4000000000ull;    // drain after a timed-out wait

__device__ __forceinline__ uint32_t swz(int row, int col) {
  // byte offset of element (row, col) inside a swizzled 64-column block set
  return (uint32_t)((col >> 6) * kSmallBlockBytes + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    ((col & 7) << 1));
}

__device__ __forceinline__ uint32_t bf16_bits(float f) {
  const __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_at(const uint8_t* base, int row, int col) {
  const uint16_t h = *reinterpret_cast<const uint16_t*>(base + swz(row, col));
  return __uint_as_float((uint32_t)h << 16);
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Non-blocking test of an mbarrier phase (try_wait may suspend the thread
// for as long as a whole small product takes, which would hide a short
// limit).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on the product barrier; on expiry records bit 0 of *err (when
// `report`) and returns false.  The limit is checked against the global
// timer and, for limits below its tick, against SM cycles (3 per ns, above
// any GB300 clock).
__device__ __noinline__ bool small_wait(uint32_t bar, uint32_t parity, int* err, uint64_t limit, bool report) {
  const uint64_t t0 = ptx::globaltimer();
  const long long c0 = clock64();
  const uint64_t cycles = limit > ~0ull / 3 ? ~0ull : 3 * limit;
  while (!mbar_test(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit || (uint64_t)(clock64() - c0) > cycles) {
      if (report) atomicOr(err, 1);
      return false;
    }
  }
  return true;
}

// One product D[tmem] = sum over kb K blocks of A_kb * B_kb (16-wide K
// steps), issued by thread 0.  Returns true, block-uniformly, once every
// thread has seen it complete; false when a wait ran out, after the
// product's MMAs have drained (bounded) so that TMEM and shared memory can
// be released.
struct Product {
  uint32_t a_base, b_base;   // shared addresses of the operands' block 0
  int k_blocks;              // 64-wide K blocks
  bool b_mn_major;           // B operand K along rows (MN-major)
  int n;                     // N of the product (multiple of 64, <= 512)
};

__device__ bool run_product(const Product& p, uint32_t tmem, uint32_t bar, uint32_t& phase, int* err,
                            uint64_t limit) {
  if (threadIdx.x == 0) {
    ptx::tc_fence_after();
    for (int n0 = 0; n0 < p.n; n0 += 256) {
      const int nn = min(256, p.n - n0);
      const uint32_t idesc = ptx::idesc_bf16(128, nn, p.b_mn_major ? 1 : 0);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = ptx::desc_sw128(p.a_base + kb * kSmallBlockBytes + kk * 32, 16, 1024);
          uint64_t bd;
          if (p.b_mn_major)  // K rows kb*64 + kk*16 of every 64-column block of X
            bd = ptx::desc_sw128(p.b_base + (n0 >> 6) * kSmallBlockBytes + (kb * 64 + kk * 16) * 128,
                                 kSmallBlockBytes, 1024);
          else               // rows 0..nn-1 of the B operand (K-major)
            bd = ptx::desc_sw128(p.b_base + kb * kSmallBlockBytes + kk * 32, 16, 1024);
          ptx::mma_bf16(tmem + n0, ad, bd, idesc, (kb | kk) != 0);
        }
      }
    }
    ptx::mma_commit(bar);
  }
  bool ok = mbar_test(bar, phase) || small_wait(bar, phase, err, limit, true);
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    if (threadIdx.x == 0) small_wait(bar, phase, err, kSmallDrainNs, false);
    __syncthreads();
  }
  phase ^= 1u;
  ptx::tc_fence_after();
  return ok;
}

// Momentum, Nesterov input and sum of squares of one element; writes the
// element of X0 = bf16(U) (or of U^T).
struct MomCtx {
  uint8_t* X;
  int cols;
  bool tr, ns_only, nesterov;
  float mu;
};

__device__ __forceinline__ float mom_elem(const MomCtx& c, int e, float g, float m_old, float& m_new) {
  float u;
  if (c.ns_only) {
    u = g;
  } else {
    m_new = fmaf(c.mu, m_old, g);
    u = c.nesterov ? fmaf(c.mu, m_new, g) : m_new;
  }
  const int r = e / c.cols, col = e - r * c.cols;
  *reinterpret_cast<uint16_t*>(c.X + (c.tr ? swz(col, r) : swz(r, col))) = (uint16_t)bf16_bits(u);
  return u;
}

__global__ void __launch_bounds__(128, 1) ns_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* X = base;                                  // 128 x 512 bf16, 8 blocks
  uint8_t* A = base + 8 * kSmallBlockBytes;           // 128 x 128 bf16, 2 blocks
  uint8_t* B = A + 2 * kSmallBlockBytes;              // 128 x 128 bf16, 2 blocks
  uint64_t* bar = reinterpret_cast<uint64_t*>(B + 2 * kSmallBlockBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // 4 floats

  const int tid = threadIdx.x;
  const SmallDesc d = a.descs[blockIdx.x];
  const MatPtrs p = a.ptrs[d.idx];
  const int64_t rows = d.rows, cols = d.cols;
  const bool tr = rows > cols;
  const int m = (int)(tr ? cols : rows), n = (int)(tr ? rows : cols);
  const int n_pad = (n + 63) & ~63;

  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(bar), 1);
    ptx::fence_mbar_init();
  }
  if (tid < 32) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  // Zero X (padding rows/columns must read as zero), A and B.
  for (int off = tid * 16; off < 12 * kSmallBlockBytes; off += 128 * 16)
    *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t phase = 0;
  bool ok = true;

  // ---- momentum, Nesterov input, X0 = bf16(U or U^T), sum of squares.
  // rows * cols <= 65536; G, M and W are 16-byte aligned (checked on the
  // host), so the body runs on float4 with four loads of each in flight.
  float ss = 0.f;
  const int total = (int)(rows * cols);
  const MomCtx mc{X, (int)cols, tr, a.ns_only != 0, a.nesterov != 0, a.mu};
  {
    const int nv = total >> 2;
    const float4* G4 = reinterpret_cast<const float4*>(p.G);
    float4* M4 = reinterpret_cast<float4*>(p.M);
    for (int v0 = tid; v0 < nv; v0 += 4 * 128) {
      float4 g[4], mo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = v0 + q * 128;
        if (v < nv) {
          g[q] = G4[v];
          mo[q] = a.ns_only ? make_float4(0.f, 0.f, 0.f, 0.f) : M4[v];
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = v0 + q * 128;
        if (v < nv) {
          float4 mn;
          const float u0 = mom_elem(mc, 4 * v + 0, g[q].x, mo[q].x, mn.x);
          const float u1 = mom_elem(mc, 4 * v + 1, g[q].y, mo[q].y, mn.y);
          const float u2 = mom_elem(mc, 4 * v + 2, g[q].z, mo[q].z, mn.z);
          const float u3 = mom_elem(mc, 4 * v + 3, g[q].w, mo[q].w, mn.w);
          ss = fmaf(u0, u0, ss); ss = fmaf(u1, u1, ss); ss = fmaf(u2, u2, ss); ss = fmaf(u3, u3, ss);
          if (!a.ns_only) M4[v] = mn;
        }
      }
    }
    for (int e = 4 * nv + tid; e < total; e += 128) {
      float mn = 0.f;
      const float u = mom_elem(mc, e, p.G[e], a.ns_only ? 0.f : p.M[e], mn);
      ss = fmaf(u, u, ss);
      if (!a.ns_only) p.M[e] = mn;
    }
  }
  // fixed-order block sum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  fence_async_smem();
  __syncthreads();
  const double tot = (double)red[0] + (double)red[1] + (double)red[2] + (double)red[3];
  const bool finite = isfinite(tot);
  const float s = finite ? (float)(1.0 / (sqrt(tot) + (double)a.eps)) : 0.f;
  if (tid == 0 && !finite) a.flags[d.idx] |= 1;

  const uint32_t xs = ptx::smem_addr(X), as = ptx::smem_addr(A), bs = ptx::smem_addr(B);
  const uint32_t bar_a = ptx::smem_addr(bar);
  const int i = tid;  // this thread's row (TMEM lane)
  const uint32_t tq = tmem + ((uint32_t)((tid >> 5) * 32) << 16);
  const float coef = a.lr * d.scale;
  const uint64_t limit = a.timeout_ns ? a.timeout_ns : kSmallTimeoutNs;

  for (int k = 0; ok && k < a.ns_steps; ++k) {
    const float ca = a.coeffs[k][0], cb = a.coeffs[k][1], cc = a.coeffs[k][2];
    const bool first = k == 0;
    const bool last = k == a.ns_steps - 1;
    // A = X X^T (K = n_pad)
    ok = run_product(Product{xs, xs, n_pad >> 6, false, 128}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    {
      const float alpha = first ? s * s : 1.f;
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tq + c0, v);
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 w;
          w.x = bf16_bits(__uint_as_float(v[j]) * alpha) | (bf16_bits(__uint_as_float(v[j + 1]) * alpha) << 16);
          w.y = bf16_bits(__uint_as_float(v[j + 2]) * alpha) | (bf16_bits(__uint_as_float(v[j + 3]) * alpha) << 16);
          w.z = bf16_bits(__uint_as_float(v[j + 4]) * alpha) | (bf16_bits(__uint_as_float(v[j + 5]) * alpha) << 16);
          w.w = bf16_bits(__uint_as_float(v[j + 6]) * alpha) | (bf16_bits(__uint_as_float(v[j + 7]) * alpha) << 16);
          *reinterpret_cast<uint4*>(A + swz(i, c0 + j)) = w;
        }
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
    // B = b A + c A A (K = 128)
    ok = run_product(Product{as, as, 2, false, 128}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tq + c0, v);
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cj = c0 + j + 2 * q;
          const float lo = fmaf(cc, __uint_as_float(v[j + 2 * q]), cb * bf16_at(A, i, cj));
          const float hi = fmaf(cc, __uint_as_float(v[j + 2 * q + 1]), cb * bf16_at(A, i, cj + 1));
          w[q] = bf16_bits(lo) | (bf16_bits(hi) << 16);
        }
        *reinterpret_cast<uint4*>(B + swz(i, c0 + j)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
    // X' = a X + B X (M = 128, N = n_pad, K = 128; X as the MN-major operand)
    ok = run_product(Product{bs, xs, 2, true, n_pad}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    const float alpha = first ? s : 1.f;
    for (int c0 = 0; c0 < n_pad; c0 += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tq + c0, v);
      if (!last) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cj = c0 + j + 2 * q;
            const float lo = alpha * fmaf(ca, bf16_at(X, i, cj), __uint_as_float(v[j + 2 * q]));
            const float hi = alpha * fmaf(ca, bf16_at(X, i, cj + 1), __uint_as_float(v[j + 2 * q + 1]));
            w[q] = bf16_bits(lo) | (bf16_bits(hi) << 16);
          }
          *reinterpret_cast<uint4*>(X + swz(i, c0 + j)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else if (i < m) {
        // O = a X + B X in fp32, straight to W (or to the output).  Row i
        // of O is row i of W (float4 read-modify-write when the row is
        // 16-byte aligned) or column i of W (lanes write neighbours).
        const bool vec = !tr && (cols & 3) == 0;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const int cj = c0 + j;
          if (cj >= n) break;
          float o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) o[q] = alpha * fmaf(ca, bf16_at(X, i, cj + q), __uint_as_float(v[j + q]));
          if (vec) {
            float4* w4 = reinterpret_cast<float4*>(p.W + (int64_t)i * cols + cj);
            float4 w = a.ns_only ? make_float4(0.f, 0.f, 0.f, 0.f) : *w4;
            if (!a.ns_only) {
              w.x = fmaf(a.decay, w.x, -coef * o[0]);
              w.y = fmaf(a.decay, w.y, -coef * o[1]);
              w.z = fmaf(a.decay, w.z, -coef * o[2]);
              w.w = fmaf(a.decay, w.w, -coef * o[3]);
            } else {
              w = make_float4(o[0], o[1], o[2], o[3]);
            }
            *w4 = w;
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (cj + q < n) {
                const int64_t off = tr ? (int64_t)(cj + q) * cols + i : (int64_t)i * cols + cj + q;
                p.W[off] = a.ns_only ? o[q] : fmaf(a.decay, p.W[off], -coef * o[q]);
              }
            }
          }
        }
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
  }
  if (ok && a.ns_steps == 0) {
    // no iteration: O = s * U, with U recomputed in fp32 from G and the
    // updated momentum (the same fused multiply-adds as above)
    for (int e = tid; e < total; e += 128) {
      const float g = p.G[e];
      const float u = a.ns_only ? g : (a.nesterov ? fmaf(a.mu, p.M[e], g) : p.M[e]);
      const float o = s * u;
      p.W[e] = a.ns_only ? o : fmaf(a.decay, p.W[e], -coef * o);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (tid < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t small_configure() {
  return cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
}

cudaError_t launch_small(const SmallArgs& a, int n_mats, cudaStream_t s) {
  ns_small_kernel<<<n_mats, 128, kSmallSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dmuon
