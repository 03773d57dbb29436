// Fused Muon step for small matrices: one CTA runs a matrix's whole step
// -- momentum, Nesterov input, norm, ns_steps quintic Newton-Schulz
// iterations and the update -- with the iterate, A and B resident in shared
// memory and the products accumulated in TMEM.  For oriented shapes with
// m <= 128 and n <= 512 (DMuon "Quick Start": TinyMLP projections at small
// widths; 64x256 tensor-parallel shards): X is at most 128 x 512 fp16 =
// 128 KB, A and B 32 KB each.
//
// DMuon "API Reference", section "direct_newton_schulz": per step
//   A = X X^T,  B = b A + c A A,  X = a X + B X,
// computed here as X = Z X with Z = a I + B stored in fp16 (the a X term
// rides in the product; no epilogue pass over X is needed).  The operands are
// fp16 with power-of-two scales (X0 = p U with p from the block's max |U|,
// later X as beta X, A as kappa X X^T), as on the chunked path.
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
// 256 threads (8 warps).  Streaming phases (momentum pass, update) use all
// of them with several 16-byte loads in flight per thread.  In the
// epilogues warp w reads TMEM lanes 32*(w%4).. (its rows) and takes half of
// the columns (w/4).  Thread 0 issues the MMAs (M = 128, fp32 accumulate,
// fp16 operands); every product completes on one mbarrier with a bounded
// wait.
#include "common.cuh"
#include "ptx.cuh"
#include "small.cuh"

namespace dmuon {

namespace {

constexpr int kThreads = kSmallThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kInFlight = 8;                          // 16-byte loads per array per thread
constexpr uint64_t kSmallTimeoutNs = 4000000000ull;  // default product wait limit
constexpr uint64_t kSmallDrainNs = 4000000000ull;    // drain after a timed-out wait

__device__ __forceinline__ uint32_t swz(int row, int col) {
  // byte offset of element (row, col) inside a swizzled 64-column block set
  return (uint32_t)((col >> 6) * kSmallBlockBytes + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    ((col & 7) << 1));
}

__device__ __forceinline__ uint32_t h_bits(float f) {
  const __half b = __float2half_rn(f);
  return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ uint32_t pack_h(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Eight consecutive fp16 of one row (col % 8 == 0): one 16-byte chunk.
__device__ __forceinline__ void load8(const uint8_t* base, int row, int col, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(base + swz(row, col));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

__device__ __forceinline__ void store8(uint8_t* base, int row, int col, const float (&f)[8]) {
  *reinterpret_cast<uint4*>(base + swz(row, col)) =
      make_uint4(pack_h(f[0], f[1]), pack_h(f[2], f[3]), pack_h(f[4], f[5]), pack_h(f[6], f[7]));
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
// steps), issued by thread 0.  Returns true, block-uniformly, once the
// product is complete (thread 0 saw its mbarrier phase, then a block
// barrier and the tcgen05 after-sync fence order every thread's TMEM reads
// after it); false when the wait ran out, after the product's MMAs have
// drained (bounded) so that TMEM and shared memory can be released.
struct Product {
  uint32_t a_base, b_base;   // shared addresses of the operands' block 0
  int k_blocks;              // 64-wide K blocks
  bool b_mn_major;           // B operand K along rows (MN-major)
  int n;                     // N of the product (multiple of 64, <= 512)
};

__device__ bool run_product(const Product& p, uint32_t tmem, uint32_t bar, uint32_t& phase, int* err,
                            uint64_t limit) {
  bool ok = true;
  if (threadIdx.x == 0) {
    ptx::tc_fence_after();
    // Descriptors are built once and advanced by their start-address field
    // (16-byte units; every operand lies below 256 KB, so no carry leaves it).
    const uint64_t a0 = ptx::desc_sw128(p.a_base, 16, 1024);
    const uint64_t b0 = p.b_mn_major ? ptx::desc_sw128(p.b_base, kSmallBlockBytes, 1024)
                                     : ptx::desc_sw128(p.b_base, 16, 1024);
    for (int n0 = 0; n0 < p.n; n0 += 256) {
      const int nn = min(256, p.n - n0);
      const uint32_t idesc = ptx::idesc_f16(128, nn, p.b_mn_major ? 1 : 0);
      // MN-major B (X): K rows kb*64 + kk*16 of every 64-column block from
      // block n0/64; K-major B: rows 0..nn-1, K columns kb*64 + kk*16.
      const uint64_t bn = b0 + (uint64_t)((n0 >> 6) * (kSmallBlockBytes >> 4));
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const uint64_t ak = a0 + (uint64_t)(kb * (kSmallBlockBytes >> 4));
        const uint64_t bk = p.b_mn_major ? bn + (uint64_t)(kb * (64 * 128 >> 4))
                                         : b0 + (uint64_t)(kb * (kSmallBlockBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16(tmem + n0, ak + 2 * kk, bk + (p.b_mn_major ? 128 * kk : 2 * kk), idesc, (kb | kk) != 0);
      }
    }
    ptx::mma_commit(bar);
    // Only the issuing thread polls; the other warps sleep in the barrier
    // below instead of taking issue slots.  On a timeout it drains the
    // product's MMAs (bounded) before anyone releases TMEM.
    ok = mbar_test(bar, phase) || small_wait(bar, phase, err, limit, true);
    if (!ok) small_wait(bar, phase, err, kSmallDrainNs, false);
  }
  ok = __syncthreads_and(ok) != 0;
  phase ^= 1u;
  ptx::tc_fence_after();
  return ok;
}

// Momentum and Nesterov input of one element: returns U, writes the new
// momentum to m_new (unless ns_only).
__device__ __forceinline__ float mom_u(const SmallArgs& a, float g, float m_old, float& m_new) {
  if (a.ns_only) return g;
  m_new = fmaf(a.mu, m_old, g);
  return a.nesterov ? fmaf(a.mu, m_new, g) : m_new;
}

// U from G and the already updated momentum (the second pass).
__device__ __forceinline__ float nest_u(const SmallArgs& a, float g, float m_new) {
  if (a.ns_only) return g;
  return a.nesterov ? fmaf(a.mu, m_new, g) : m_new;
}

// The two passes over G and M.  Pass 0: M <- mu*M + G and U; returns this
// thread's max |U| (NaN inputs set *nan).  Pass 1: U again from G and the
// updated M (the same fused multiply-adds, so the same U), X0 = fp16(p U)
// (or p U^T) into shared memory; returns this thread's sum of (p U)^2 in a
// fixed order.  The power of two p comes from the block's max |U| between
// the passes, so p U never leaves fp16's normal range whatever the input's
// scale.  Rows of 4k floats go as float4 (G, M, W are 16-byte aligned);
// (row, column) advance incrementally, no division per element.
__device__ float momentum_pass(const SmallArgs& a, const MatPtrs& p, uint8_t* X, int rows, int cols, bool tr,
                               int pass, float ps, bool* nan) {
  const int tid = threadIdx.x;
  float acc = 0.f;
  bool bad = false;
  auto take = [&](float u) {
    if (pass == 0) {
      acc = fmaxf(acc, fabsf(u));
      bad |= u != u;
      return 0.f;
    }
    const float x = u * ps;
    acc = fmaf(x, x, acc);
    return x;
  };
  if ((cols & 3) == 0) {
    const int c4n = cols >> 2, total4 = rows * c4n;
    const int dr = kThreads / c4n, dc = kThreads % c4n;
    int r = tid / c4n, c = tid % c4n;
    const float4* G4 = reinterpret_cast<const float4*>(p.G);
    float4* M4 = reinterpret_cast<float4*>(p.M);
    for (int v0 = tid; v0 < total4; v0 += kInFlight * kThreads) {
      float4 g[kInFlight], mo[kInFlight];
      int rr[kInFlight], cc[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kThreads;
        rr[k] = r;
        cc[k] = c;
        g[k] = mo[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < total4) {
          g[k] = G4[v];
          if (!a.ns_only) mo[k] = M4[v];
        }
        r += dr;
        c += dc;
        if (c >= c4n) { c -= c4n; ++r; }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kThreads;
        if (v < total4) {
          float u[4];
          if (pass == 0) {
            float4 mn = make_float4(0.f, 0.f, 0.f, 0.f);
            u[0] = mom_u(a, g[k].x, mo[k].x, mn.x);
            u[1] = mom_u(a, g[k].y, mo[k].y, mn.y);
            u[2] = mom_u(a, g[k].z, mo[k].z, mn.z);
            u[3] = mom_u(a, g[k].w, mo[k].w, mn.w);
            if (!a.ns_only) M4[v] = mn;
          } else {
            u[0] = nest_u(a, g[k].x, mo[k].x);
            u[1] = nest_u(a, g[k].y, mo[k].y);
            u[2] = nest_u(a, g[k].z, mo[k].z);
            u[3] = nest_u(a, g[k].w, mo[k].w);
          }
          float x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) x[j] = take(u[j]);
          if (pass == 1) {
            const int col = 4 * cc[k];
            if (!tr) {
              *reinterpret_cast<uint2*>(X + swz(rr[k], col)) = make_uint2(pack_h(x[0], x[1]), pack_h(x[2], x[3]));
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) *reinterpret_cast<uint16_t*>(X + swz(col + j, rr[k])) = (uint16_t)h_bits(x[j]);
            }
          }
        }
      }
    }
  } else {
    const int total = rows * cols;
    const int dr = kThreads / cols, dc = kThreads % cols;
    int r = tid / cols, c = tid % cols;
    for (int e0 = tid; e0 < total; e0 += kInFlight * kThreads) {
      float g[kInFlight], mo[kInFlight];
      int rr[kInFlight], cc[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int e = e0 + k * kThreads;
        rr[k] = r;
        cc[k] = c;
        g[k] = mo[k] = 0.f;
        if (e < total) {
          g[k] = p.G[e];
          if (!a.ns_only) mo[k] = p.M[e];
        }
        r += dr;
        c += dc;
        if (c >= cols) { c -= cols; ++r; }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int e = e0 + k * kThreads;
        if (e < total) {
          float u;
          if (pass == 0) {
            float mn = 0.f;
            u = mom_u(a, g[k], mo[k], mn);
            if (!a.ns_only) p.M[e] = mn;
          } else {
            u = nest_u(a, g[k], mo[k]);
          }
          const float x = take(u);
          if (pass == 1)
            *reinterpret_cast<uint16_t*>(X + (tr ? swz(cc[k], rr[k]) : swz(rr[k], cc[k]))) = (uint16_t)h_bits(x);
        }
      }
    }
  }
  if (bad) *nan = true;
  return acc;
}

struct FinalCtx {
  float alpha, coef, decay;
  int m, n, cols;
  bool ns_only;
};

// Last iteration, transposed matrix (W is n x m): row `row` of O is column
// `row` of W, so the lanes of a warp write neighbouring addresses.  Columns
// [c_lo, c_hi) of this thread's half, 32 per TMEM load, W loads issued
// before the stores.
__device__ __forceinline__ void final_transposed(const FinalCtx& f, float* W, uint32_t tq, int row, int c_lo,
                                                 int c_hi) {
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    uint32_t v[32];
    ptx::tmem_ld32(tq + c0, v);
    if (row < f.m) {
      float w[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        w[j] = (!f.ns_only && c0 + j < f.n) ? W[(int64_t)(c0 + j) * f.cols + row] : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int cj = c0 + j;
        if (cj < f.n) {
          const float o = f.alpha * __uint_as_float(v[j]);
          W[(int64_t)cj * f.cols + row] = f.ns_only ? o : fmaf(f.decay, w[j], -f.coef * o);
        }
      }
    }
  }
}

// Last iteration, row-major matrix: O goes through a 128 x 128 fp32 staging
// tile (the A and B regions, free after the last product) with 16-byte
// chunks swizzled by row, then whole rows of W are updated by one warp each
// (coalesced 512-byte rows, 16 rows' loads in flight per warp).
__device__ __forceinline__ void final_rows(const FinalCtx& f, float* W, uint32_t tq, float* stg, int row, int h,
                                           int n_pad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = (f.cols & 3) == 0;
  for (int p0 = 0; p0 < n_pad; p0 += 128) {
#pragma unroll
    for (int hc = 0; hc < 64; hc += 32) {
      const int c0 = p0 + 64 * h + hc;
      if (c0 < n_pad) {
        uint32_t v[32];
        ptx::tmem_ld32(tq + c0, v);
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          float o[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) o[t] = f.alpha * __uint_as_float(v[j + t]);
          const int ch = (c0 - p0 + j) >> 2;
          *reinterpret_cast<float4*>(stg + row * 128 + ((ch ^ (row & 31)) << 2)) = make_float4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<float4*>(stg + row * 128 + (((ch + 1) ^ (row & 31)) << 2)) =
              make_float4(o[4], o[5], o[6], o[7]);
        }
      }
    }
    __syncthreads();
    const int cl = p0 + 4 * lane;
    float4 w[128 / kWarps];
#pragma unroll
    for (int k = 0; k < 128 / kWarps; ++k) {
      const int r = warp + kWarps * k;
      w[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!f.ns_only && r < f.m && cl < f.n) {
        const float* src = W + (int64_t)r * f.cols + cl;
        if (vec) {
          w[k] = *reinterpret_cast<const float4*>(src);
        } else {
          w[k].x = src[0];
          if (cl + 1 < f.n) w[k].y = src[1];
          if (cl + 2 < f.n) w[k].z = src[2];
          if (cl + 3 < f.n) w[k].w = src[3];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 128 / kWarps; ++k) {
      const int r = warp + kWarps * k;
      if (r < f.m && cl < f.n) {
        const float4 o = *reinterpret_cast<const float4*>(stg + r * 128 + ((lane ^ (r & 31)) << 2));
        float4 u;
        if (f.ns_only) {
          u = o;
        } else {
          u.x = fmaf(f.decay, w[k].x, -f.coef * o.x);
          u.y = fmaf(f.decay, w[k].y, -f.coef * o.y);
          u.z = fmaf(f.decay, w[k].z, -f.coef * o.z);
          u.w = fmaf(f.decay, w[k].w, -f.coef * o.w);
        }
        float* dst = W + (int64_t)r * f.cols + cl;
        if (vec) {
          *reinterpret_cast<float4*>(dst) = u;
        } else {
          dst[0] = u.x;
          if (cl + 1 < f.n) dst[1] = u.y;
          if (cl + 2 < f.n) dst[2] = u.z;
          if (cl + 3 < f.n) dst[3] = u.w;
        }
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1) ns_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* X = base;                                  // 128 x 512 fp16, 8 blocks
  uint8_t* A = base + 8 * kSmallBlockBytes;           // 128 x 128 fp16, 2 blocks
  uint8_t* B = A + 2 * kSmallBlockBytes;              // 128 x 128 fp16, 2 blocks
  uint64_t* bar = reinterpret_cast<uint64_t*>(B + 2 * kSmallBlockBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // kWarps floats

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = warp >> 2;                 // column half in the epilogues
  const int row = 32 * (warp & 3) + lane;  // TMEM lane = row of X, A, B
  const SmallDesc d = a.descs[blockIdx.x];
  const MatPtrs p = a.ptrs[d.idx];
  const int rows = (int)d.rows, cols = (int)d.cols;
  const bool tr = rows > cols;
  const int m = tr ? cols : rows, n = tr ? rows : cols;
  const int n_pad = (n + 63) & ~63;
  // m x m products are m_pad wide (64 or 128); their epilogues write all 128
  // rows of columns < m_pad and nothing reads a column >= m_pad
  const int m_pad = (m + 63) & ~63, hw = m_pad >> 1;
  const uint32_t tcols = n_pad <= 128 ? 128u : (n_pad <= 256 ? 256u : 512u);

  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(bar), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), tcols);
    ptx::tmem_relinquish();
  }
  // Zero the X blocks in use (padding rows/columns must read as zero); A and
  // B are written whole by their epilogues before they are read.
  for (int off = tid * 16; off < (n_pad >> 6) * kSmallBlockBytes; off += kThreads * 16)
    *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  uint32_t phase = 0;
  bool ok = true;

  // ---- momentum and Nesterov input: max |U| first, then p and X0 = p U with
  // the sum of squares of p U (fixed order)
  __shared__ int nan_seen;
  if (tid == 0) nan_seen = 0;
  __syncthreads();
  bool nan = false;
  float mx = momentum_pass(a, p, X, rows, cols, tr, 0, 1.f, &nan);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  if (nan) nan_seen = 1;
  __syncthreads();  // also orders this CTA's momentum stores before the second pass reads them
  mx = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red[w]);
  int ex = 0;
  frexpf(mx, &ex);
  const float ps = (mx > 0.f && !isinf(mx)) ? ldexpf(1.f, min(127, max(-126, 11 - ex))) : 1.f;
  __syncthreads();
  float ss = momentum_pass(a, p, X, rows, cols, tr, 1, ps, &nan);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  fence_async_smem();
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tot += (double)red[w];
  const bool finite = !nan_seen && !isinf(mx) && isfinite(tot);
  // s = 1 / (||U|| + eps), ||U|| = sqrt(tot) / ps; X0 holds ps U, so the first
  // products take s/ps (= 0 for a zero or non-finite input)
  const float s = (finite && mx > 0.f) ? (float)(1.0 / (sqrt(tot) / (double)ps + (double)a.eps)) : 0.f;
  const float s_x0 = (finite && mx > 0.f) ? (float)(1.0 / (sqrt(tot) + (double)a.eps * (double)ps)) : 0.f;
  if (tid == 0 && !finite) a.flags[d.idx] |= 1;
  // fp16 scales: A holds kappa X X^T, X after the first product beta' X with
  // beta' = beta / 2^floor(log2 nu) when nu = ||X0||_F = ||U|| / (||U|| + eps)
  // is below 1/2 (an input far below eps), else beta
  float beta = scale_beta(n);
  {
    const double r = sqrt(tot), nu = r / (r + (double)a.eps * (double)ps);
    if (finite && nu < 0.5 && nu > 0.0) {
      int ex = 0;
      frexp(nu, &ex);
      beta = ldexpf(beta, min(100, 1 - ex));
    }
  }
  const float kap = scale_kappa(m), ikap = 1.f / kap, ibeta = 1.f / beta;

  const uint32_t xs = ptx::smem_addr(X), as = ptx::smem_addr(A), bs = ptx::smem_addr(B);
  const uint32_t bar_a = ptx::smem_addr(bar);
  const float coef = a.lr * d.scale;
  const uint64_t limit = a.timeout_ns ? a.timeout_ns : kSmallTimeoutNs;

  for (int k = 0; ok && k < a.ns_steps; ++k) {
    const float ca = a.coeffs[k][0], cb = a.coeffs[k][1], cc = a.coeffs[k][2];
    const bool first = k == 0;
    const bool last = k == a.ns_steps - 1;
    // X = xsc * (stored X): s/p for X0 = p U, 1/beta afterwards
    const float xsc = first ? s_x0 : ibeta;
    // A = kappa xsc^2 X X^T (N = m_pad, K = n_pad)
    ok = run_product(Product{xs, xs, n_pad >> 6, false, m_pad}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    {
      const float alpha = kap * xsc * xsc;
      for (int c0 = h * hw; c0 < (h + 1) * hw; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tq + c0, v);
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          float o[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) o[t] = __uint_as_float(v[j + t]) * alpha;
          store8(A, row, c0 + j, o);
        }
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
    // Z = a I + (b/kappa) A + (c/kappa^2) A A (N = K = m_pad), stored where B lives
    ok = run_product(Product{as, as, m_pad >> 6, false, m_pad}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    const float gcc = cc * ikap * ikap, gcb = cb * ikap;
    for (int c0 = h * hw; c0 < (h + 1) * hw; c0 += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tq + c0, v);
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        float av[8], o[8];
        load8(A, row, c0 + j, av);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          o[t] = fmaf(gcc, __uint_as_float(v[j + t]), gcb * av[t]) + (c0 + j + t == row ? ca : 0.f);
        store8(B, row, c0 + j, o);
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
    // X' = beta xsc Z X stored (M = 128, N = n_pad, K = m_pad; X as the
    // MN-major operand); the last product gives O = xsc Z X in fp32
    ok = run_product(Product{bs, xs, m_pad >> 6, true, n_pad}, tmem, bar_a, phase, a.err, limit);
    if (!ok) break;
    const float alpha = last ? xsc : xsc * beta;
    const int half = n_pad >> 1;
    if (!last) {
      for (int c0 = h * half; c0 < (h + 1) * half; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tq + c0, v);
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          float x[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) x[t] = alpha * __uint_as_float(v[j + t]);
          store8(X, row, c0 + j, x);
        }
      }
    } else {
      const FinalCtx f{alpha, coef, a.decay, m, n, cols, a.ns_only != 0};
      if (tr)
        final_transposed(f, p.W, tq, row, h * half, (h + 1) * half);
      else
        final_rows(f, p.W, tq, reinterpret_cast<float*>(A), row, h, n_pad);
    }
    ptx::tc_fence_before();
    fence_async_smem();
    __syncthreads();
  }
  if (ok && a.ns_steps == 0) {
    // no iteration: O = s * U, with U recomputed in fp32 from G and the
    // updated momentum (the same fused multiply-adds as the momentum pass)
    const int total = rows * cols, total4 = total >> 2;
    const float4* G4 = reinterpret_cast<const float4*>(p.G);
    const float4* M4 = reinterpret_cast<const float4*>(p.M);
    float4* W4 = reinterpret_cast<float4*>(p.W);
    auto upd = [&](float g, float mnew, float w) {
      const float u = a.ns_only ? g : (a.nesterov ? fmaf(a.mu, mnew, g) : mnew);
      const float o = s * u;
      return a.ns_only ? o : fmaf(a.decay, w, -coef * o);
    };
    for (int v = tid; v < total4; v += kThreads) {
      const float4 g = G4[v];
      const float4 mv = a.ns_only ? make_float4(0.f, 0.f, 0.f, 0.f) : M4[v];
      const float4 w = a.ns_only ? make_float4(0.f, 0.f, 0.f, 0.f) : W4[v];
      W4[v] = make_float4(upd(g.x, mv.x, w.x), upd(g.y, mv.y, w.y), upd(g.z, mv.z, w.z), upd(g.w, mv.w, w.w));
    }
    for (int e = 4 * total4 + tid; e < total; e += kThreads)
      p.W[e] = upd(p.G[e], a.ns_only ? 0.f : p.M[e], a.ns_only ? 0.f : p.W[e]);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, tcols);
  }
}

}  // namespace

cudaError_t small_configure() {
  return cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
}

cudaError_t launch_small(const SmallArgs& a, int n_mats, cudaStream_t s) {
  ns_small_kernel<<<n_mats, kThreads, kSmallSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dmuon
