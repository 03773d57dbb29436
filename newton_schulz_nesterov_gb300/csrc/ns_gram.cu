// Gram-space Newton-Schulz phases on sm_103a: symmetric m x m products of
// one restart window (DMuon "API Reference", sections gram_newton_schulz and
// gram_newton_schulz_factors), one persistent CTA-pair launch per phase over
// every matrix of a chunk.
//
//   R~ = kappa X X^T                          (fp16 X, K = n; first of a window)
//   Z  = a I + (b/kappa) R~ + (c/kappa^2) R~ R~   (two buffers alternating by step;
//                                                 a window's first Q is its Z)
//   Q' = Z Q
//   W~ = R~ Z
//   R~' = Z W~
//
// Every operand is symmetric, so L M = L M^T: both operands are read
// K-major (rows of L and rows of M).  Only the 256x256 super-tiles on or
// above the diagonal are computed; off-diagonal tiles are also written
// transposed.  The X Q products (restart and final update) run on the
// direct path's Apply kernel with a = 0 and Q as its left operand.
//
// CTA pair (cta_group::2) as in the direct kernels: warp 0 of both CTAs
// loads operand halves by TMA into a six-stage ring completing on rank 0's
// barrier; warp 1 of rank 0 issues tcgen05.mma (M = 256, N = 256, K = 16;
// fp16 in, fp32 accumulate) into one of two TMEM accumulators;
// warps 2-5 of both CTAs run the epilogue of their 128 rows.  Every wait is
// bounded; on expiry the CTA records bit 0 of *err, drains its own copies
// and MMAs (bounded), frees TMEM and returns.
#include "common.cuh"
#include "gram.cuh"
#include "ptx.cuh"

namespace dmuon {

namespace {

constexpr uint64_t kTimeoutNs = 4000000000ull;       // default: 4 s without progress
constexpr uint64_t kDrainTimeoutNs = 4000000000ull;  // drains after an abort

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                       bool honour_abort, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try(bar, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(err, 1);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                         uint64_t limit_ns) {
  if (ptx::mbar_try(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, err, true, limit_ns);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 32 consecutive fp16 of one row -> fp32; zero outside [0, ncols) or when
// the row is invalid.  Rows start 16-byte aligned (ld % 8 == 0, c % 32 == 0).
__device__ __forceinline__ void load_row32_h(const uint16_t* rowp, int64_t c, int64_t ncols, bool row_ok,
                                             float (&f)[32]) {
  if (row_ok && c + 32 <= ncols) {
    const uint4* p = reinterpret_cast<const uint4*>(rowp + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = p[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        f[q * 8 + 2 * k] = t.x;
        f[q * 8 + 2 * k + 1] = t.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      f[j] = 0.f;
      if (row_ok && c + j < ncols) {
        const uint16_t hb = rowp[c + j];
        f[j] = __half2float(*reinterpret_cast<const __half*>(&hb));
      }
    }
  }
}

// Store 32 packed 16-bit values (16 words) at rowp[c..c+31], clipped to ncols.
__device__ __forceinline__ void store_row32(uint16_t* rowp, int64_t c, int64_t ncols, bool row_ok,
                                            const uint32_t (&w)[16]) {
  if (!row_ok) return;
  if (c + 32 <= ncols && (reinterpret_cast<uintptr_t>(rowp + c) & 31u) == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) ptx::st_global_v8(rowp + c + 16 * q, w + 8 * q);  // two whole sectors
  } else if (c + 32 <= ncols) {
    uint4* p = reinterpret_cast<uint4*>(rowp + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c + j < ncols) rowp[c + j] = (uint16_t)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
  }
}

// Store only entries j in [lo, hi) of 32 packed 16-bit values at
// rowp[c + j], clipped to ncols.
__device__ __forceinline__ void store_row32_part(uint16_t* rowp, int64_t c, int64_t ncols, bool row_ok,
                                                 const uint32_t (&w)[16], int lo, int hi) {
  if (!row_ok) return;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j >= lo && j < hi && c + j < ncols)
      rowp[c + j] = (uint16_t)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
}

// Mirror store of a 32x32 block of 16-bit values held one row per lane:
// lane L writes column L of the block as row (c + L) of the destination,
// columns [rbase, rbase+32) clipped to n_lim, through the warp's 32x17-word
// scratch.  strict_upper: write only the entries that came from above the
// block's diagonal (columns < L of row c + L), for a block on the diagonal.
__device__ __forceinline__ void mirror_store32(uint16_t* base, int64_t ld, int64_t c, int64_t rbase,
                                               int64_t n_lim, int lane, const uint32_t (&w)[16],
                                               uint32_t* scratch, bool strict_upper = false) {
#pragma unroll
  for (int k = 0; k < 16; ++k) scratch[lane * 17 + k] = w[k];
  __syncwarp();
  uint32_t t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t w0 = scratch[(2 * i) * 17 + (lane >> 1)];
    const uint32_t w1 = scratch[(2 * i + 1) * 17 + (lane >> 1)];
    const uint32_t h0 = (lane & 1) ? (w0 >> 16) : (w0 & 0xFFFFu);
    const uint32_t h1 = (lane & 1) ? (w1 >> 16) : (w1 & 0xFFFFu);
    t[i] = h0 | (h1 << 16);
  }
  __syncwarp();
  const int64_t dr = c + lane;
  if (strict_upper)
    store_row32_part(base + dr * ld, rbase, n_lim, dr < n_lim, t, 0, lane);
  else
    store_row32(base + dr * ld, rbase, n_lim, dr < n_lim, t);
}

// Writes one 32x32 block of a symmetric result.  Off-diagonal super-tiles:
// the block and its mirror.  Diagonal super-tiles are made exactly
// symmetric from their upper triangle: blocks above the diagonal are
// written with their mirror, blocks below are skipped (their mirror comes
// from above), a block on the diagonal keeps its upper entries and mirrors
// the strictly upper ones.  Products of the Gram-space factors assume their
// operands symmetric (L M^T = L M); a diagonal tile left as computed is
// symmetric only to rounding, and that antisymmetric part grows step after
// step within a window.
__device__ __forceinline__ void store_sym_block(uint16_t* dst, int64_t ld, int64_t r, int64_t c, int64_t rbase,
                                                int64_t m, bool row_ok, bool diag_tile, bool off_mirror, int lane,
                                                const uint32_t (&w)[16], uint32_t* scratch) {
  if (!diag_tile) {
    store_row32(dst + r * ld, c, m, row_ok, w);
    if (off_mirror) mirror_store32(dst, ld, c, rbase, m, lane, w, scratch);
  } else if (c > rbase) {
    store_row32(dst + r * ld, c, m, row_ok, w);
    mirror_store32(dst, ld, c, rbase, m, lane, w, scratch);
  } else if (c == rbase) {
    store_row32_part(dst + r * ld, c, m, row_ok, w, lane, 32);
    mirror_store32(dst, ld, c, rbase, m, lane, w, scratch, true);
  }
}

// Epilogue of one 128-row half of a 256x256 super-tile (item.y already the
// 128-row tile of this rank).
__device__ __forceinline__ float kappa_pow(const GramDesc& g, int p) {
  float f = 1.f;
  for (int i = 0; i < p; ++i) f *= g.kappa;
  for (int i = 0; i < -p; ++i) f *= g.inv_kappa;
  return f;
}

__device__ __forceinline__ void gram_epilogue(const GramArgs& a, const int4 item, uint32_t tacc, int quad, int lane,
                                              uint32_t* scratch) {
  const GramDesc& g = a.gd[item.x];
  const int64_t m = g.m, ld = g.ld;
  const int64_t row0 = (int64_t)item.y * kBM;
  const int64_t col0 = (int64_t)item.z * kBN;
  const int64_t rbase = row0 + quad * 32;
  const int64_t r = rbase + lane;
  const bool row_ok = r < m;
  const uint32_t tq = tacc + ((uint32_t)(quad * 32) << 16);
  const bool mirror = (item.y >> 1) < item.z;
  const bool diag_tile = (item.y >> 1) == item.z;
  float gs = a.g0 * kappa_pow(g, a.gpow);
  if (a.xscale == 1) {
    const float s = a.svec[item.x];
    gs *= s * s;
  } else if (a.xscale == 2) {
    const float ib = 1.f / a.bvec[item.x];
    gs *= ib * ib;
  }
  const float c1 = a.c1 * kappa_pow(g, a.p1pow);
  const uint16_t* p1 = a.add1 >= 0 ? g.buf[a.add1] : nullptr;
  uint16_t* dst = g.buf[a.out];
  uint16_t* dst2 = a.out2 >= 0 ? g.buf[a.out2] : nullptr;
#pragma unroll 1
  for (int ch = 0; ch < kBN / 32; ++ch) {
    const int64_t c = col0 + ch * 32;
    if (c >= m) break;  // warp-uniform
    uint32_t v[32];
    ptx::tmem_ld32(tq + ch * 32, v);
    float f[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = gs * __uint_as_float(v[j]);
    if (p1) {
      float t[32];
      load_row32_h(p1 + r * ld, c, m, row_ok, t);
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = fmaf(c1, t[j], f[j]);
    }
    if (a.diag != 0.f) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (r == c + j) f[j] += a.diag;
    }
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = pack_f16(f[2 * k], f[2 * k + 1]);
    store_sym_block(dst, ld, r, c, rbase, m, row_ok, diag_tile, mirror, lane, w, scratch);
    if (dst2)  // the same values into a second buffer
      store_sym_block(dst2, ld, r, c, rbase, m, row_ok, diag_tile, mirror, lane, w, scratch);
  }
}

struct PairSmem {
  uint8_t* stages;     // kPairStages x (A half 16 KB | B half 16 KB), 1024-aligned
  uint32_t* scratch;   // 4 warps x 32 x 17 words
  uint64_t* bars;      // full[6], empty[6], tfull[2], tempty[2], drain
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ PairSmem carve_pair(uint8_t* raw) {
  PairSmem s;
  const uint32_t a = ptx::smem_addr(raw);
  uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
  s.stages = base;
  uint8_t* after = base + kPairStages * kPairStageBytes;
  s.scratch = reinterpret_cast<uint32_t*>(after);
  s.bars = reinterpret_cast<uint64_t*>(after + 4 * kEpiWords * 4);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + 2 * kPairStages + 5);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  return s;
}

// XOP = 1: operands are X[src]; XOP = 0: buf[opA], buf[opB] (both fp16).
template <int XOP>
__global__ void __launch_bounds__(kGemmThreads, 1) ns_gram_pair_kernel(const __grid_constant__ GramArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const PairSmem sm = carve_pair(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns ? a.timeout_ns : kTimeoutNs;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const WorkRange wr = work_range(a.starts, pair, npairs, a.n_items);

  uint64_t* full = sm.bars;
  uint64_t* empty = sm.bars + kPairStages;
  uint64_t* tfull = sm.bars + 2 * kPairStages;
  uint64_t* tempty = sm.bars + 2 * kPairStages + 2;
  uint64_t* drain = sm.bars + 2 * kPairStages + 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(full + s), 1);
      ptx::mbar_init(ptx::smem_addr(empty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(tfull + i), 1);
      ptx::mbar_init(ptx::smem_addr(tempty + i), 8);  // 4 epilogue warps x 2 ranks
    }
    ptx::mbar_init(ptx::smem_addr(drain), 1);
    *sm.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {  // one warp of each rank allocates the pair's TMEM together
    ptx::tmem_alloc_pair(ptx::smem_addr(sm.tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both ranks' barriers exist before any remote signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t it = 0;
      bool ok = true;
      for (int w = wr.w0; ok && w < wr.w1; w += wr.step) {
        const int4 item = a.items[w];
        const CUtensorMap* mapA;
        const CUtensorMap* mapB;
        if (XOP) {
          mapA = mapB = a.xmaps + (size_t)item.x * kMapsPerMat + a.src;
        } else {
          const CUtensorMap* g = a.gmaps + (size_t)item.x * kGramBufs;
          mapA = g + a.opA;
          mapB = g + a.opB;
        }
        const int rowA = item.y * 256 + (int)rank * 128;
        const int rowB = item.z * 256 + (int)rank * 128;
        for (int kb = 0; kb < item.w; ++kb, ++it) {
          const uint32_t s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1u;
          if (!wait_bar(ptx::smem_addr(empty + s), ph ^ 1u, sm.abort_flag, a.err, tmo)) { ok = false; break; }
          const uint32_t fb_local = ptx::smem_addr(full + s);
          const uint32_t fb = ptx::mapa_shared(fb_local, 0);
          if (leader) ptx::mbar_expect_tx(fb_local, 2 * kPairStageBytes);
          const uint32_t sa = ptx::smem_addr(sm.stages + s * kPairStageBytes);
          const uint32_t sb = sa + kPairHalfBytes;
          const int k0 = kb * kBK;
          ptx::tma_load_2d_pair(sa, mapA, k0, rowA, fb);
          ptx::tma_load_2d_pair(sa + kBoxBytes, mapA, k0, rowA + kBox, fb);
          ptx::tma_load_2d_pair(sb, mapB, k0, rowB, fb);
          ptx::tma_load_2d_pair(sb + kBoxBytes, mapB, k0, rowB + kBox, fb);
        }
      }
      if (leader && (!ok || *sm.abort_flag)) {
        // Drain: the last issued stages' bytes (both ranks') must land before
        // exit; bounded, ignoring the abort flag.
        const uint32_t n_out = it < (uint32_t)kPairStages ? it : (uint32_t)kPairStages;
        for (uint32_t i = it - n_out; i < it; ++i)
          wait_slow(ptx::smem_addr(full + (i % kPairStages)), (i / kPairStages) & 1u, sm.abort_flag, a.err, false,
                    kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_f16(256, kBN, 0);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      bool issued = false;
      for (int w = wr.w0; ok && w < wr.w1; w += wr.step, ++tc) {
        const int4 item = a.items[w];
        const uint32_t acc = tc & 1u;
        if (!wait_bar(ptx::smem_addr(tempty + acc), ((tc >> 1) & 1u) ^ 1u, sm.abort_flag, a.err, tmo)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + acc * kBN;
        for (int kb = 0; kb < item.w; ++kb, ++it) {
          const uint32_t s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1u;
          if (!wait_bar(ptx::smem_addr(full + s), ph, sm.abort_flag, a.err, tmo)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(sm.stages + s * kPairStageBytes);
          const uint32_t sb = sa + kPairHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = ptx::desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = ptx::desc_sw128(sb + kk * 32, 16, 1024);
            ptx::mma_f16_pair(dt, ad, bd, idesc, (kb | kk) != 0);
          }
          issued = true;
          ptx::mma_commit_multicast(ptx::smem_addr(empty + s), 0x3);
        }
        if (!ok) break;
        ptx::mma_commit_multicast(ptx::smem_addr(tfull + acc), 0x3);
      }
      if (issued && (!ok || *sm.abort_flag)) {
        ptx::mma_commit_pair(ptx::smem_addr(drain));
        wait_slow(ptx::smem_addr(drain), 0, sm.abort_flag, a.err, false, kDrainTimeoutNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31 for this warp
    uint32_t* scratch = sm.scratch + (warp - 2) * kEpiWords;
    uint32_t tc = 0;
    for (int w = wr.w0; w < wr.w1; w += wr.step, ++tc) {
      int4 item = a.items[w];
      const uint32_t acc = tc & 1u;
      if (!wait_bar(ptx::smem_addr(tfull + acc), (tc >> 1) & 1u, sm.abort_flag, a.err, tmo)) break;
      ptx::tc_fence_after();
      item.y = item.y * 2 + (int)rank;  // this rank's 128-row tile
      gram_epilogue(a, item, tmem_base + acc * kBN, quad, lane, scratch);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_addr(tempty + acc), 0));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no rank frees TMEM or exits while its pair is busy
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int XOP>
cudaError_t launch_one(const GramArgs& a, int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ns_gram_pair_kernel<XOP>, a);
}

}  // namespace

cudaError_t gram_configure() {
  cudaError_t e = cudaFuncSetAttribute(ns_gram_pair_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(ns_gram_pair_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
}

cudaError_t launch_gram_pair(const GramArgs& a, int clusters, cudaStream_t s) {
  return a.x_operand ? launch_one<1>(a, clusters, s) : launch_one<0>(a, clusters, s);
}

}  // namespace dmuon
