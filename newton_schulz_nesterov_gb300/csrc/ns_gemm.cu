// Tensor-core phases of quintic Newton-Schulz on sm_103a (tcgen05 + TMEM +
// TMA), one persistent launch per phase over every matrix of the list.
//
// DMuon "API Reference", section "direct_newton_schulz": per step k,
//   X <- a_k X + b_k (X X^T) X + c_k (X X^T)^2 X
// computed as three products:
//   Gram   A = X X^T             symmetric, m x m, K = n
//   Gram2  B = b A + c A A       symmetric, m x m, K = m (A A = A A^T)
//   Apply  X' = a X + B X        m x n, K = m  (last step: weight update)
// The symmetric products compute only the 256x256 super-tiles on or above
// the diagonal and write the transposed copy of each off-diagonal tile, the
// tile saving the pages' SYRK kernels describe (section "newton_schulz").
//
// CTA layout (192 threads, one CTA per SM, persistent over a static run of
// work items dealt by the host, longest first to the least-loaded CTA):
//   warp 0   TMA producer: 64-wide K blocks of both operands into a
//            shared-memory ring (128-byte swizzle, 64x64 boxes)
//   warp 1   TMEM allocator and single-thread tcgen05.mma issuer
//            (M=128, N=256 or 128, K=16 per instruction, fp32 accumulate)
//   warps 2-5 epilogue: TMEM -> registers, fused scaling / a*X / b*A terms,
//            16-bit stores (direct and mirrored) or the fp32 weight update
// Single CTAs take 128 x 256 tiles (4 stages of 48 KB) or, for lists too
// small to fill the SMs, 128 x 128 tiles (6 stages of 32 KB); CTA pairs
// (cta_group::2, below) take 256 x 256 tiles.
// Operands are fp16 in the first iterations and bf16 after (kind::f16,
// fp32 accumulate); every stored buffer carries a power-of-two scale
// (MatDesc) that keeps its entries in fp16's normal range, undone in the
// epilogues.  Two accumulators in TMEM let the epilogue of one tile overlap
// the main loop of the next.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns, default 4 s without
// progress); on timeout the CTA records
// bit 0 of *err, stops issuing, drains its own copies and MMAs with bounded
// waits, frees TMEM and returns.
#include "common.cuh"
#include "ptx.cuh"

namespace dmuon {

namespace {

constexpr uint64_t kTimeoutNs = 4000000000ull;  // default: 4 s without progress
constexpr uint64_t kDrainTimeoutNs = 4000000000ull;  // drains after an abort

// Single-CTA kernel geometry for a tile of 128 rows x BN columns (BN = 256,
// or 128 for lists too small to fill the SMs with 128 x 256 tiles): B is
// BN x 64 per K block, so a stage is 48 or 32 KB and 4 or 6 stages fit.
template <int BN>
struct SingleCfg {
  static constexpr int kStageB = kABytes + BN * kBK * 2;
  static constexpr int kNStages = BN == kBN ? kStages : 6;
  static constexpr int kSmem = 1024 /*align slack*/ + kNStages * kStageB + 4 * kEpiWords * 4 + 256;
  static constexpr int kTmem = 2 * BN;  // two accumulators
};
static_assert(SingleCfg<kBN>::kSmem == kGemmSmem, "128 x 256 geometry");
static_assert(SingleCfg<128>::kSmem <= 227 * 1024, "128 x 128 geometry");

struct Smem {
  uint8_t* stages;     // stages x (A 16 KB | B BN x 64 x 2), 1024-aligned
  uint32_t* scratch;   // 4 warps x 32 x 17 words
  uint64_t* bars;      // full[stages], empty[stages], tfull[2], tempty[2], drain
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  uint32_t* tile_done;  // fused launches: epilogue warps done per accumulator slot
};

template <int BN>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  using C = SingleCfg<BN>;
  Smem s;
  const uint32_t a = ptx::smem_addr(raw);
  uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
  s.stages = base;
  s.scratch = reinterpret_cast<uint32_t*>(base + C::kNStages * C::kStageB);
  s.bars = reinterpret_cast<uint64_t*>(base + C::kNStages * C::kStageB + 4 * kEpiWords * 4);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + 2 * C::kNStages + 5);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.tile_done = s.tmem_slot + 2;
  return s;
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* err, bool honour_abort, uint64_t limit_ns) {
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err, uint64_t limit_ns) {
  if (ptx::mbar_try(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, err, true, limit_ns);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool f16) {
  if (f16) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, bool f16) {
  if (f16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// 32 consecutive 16-bit values (fp16, or bf16 when !f16) of one row -> fp32,
// zero outside [0, ncols) or when the row is invalid.
__device__ __forceinline__ void load_row32(const __half* rowp, int64_t c, int64_t ncols,
                                           bool row_ok, float (&f)[32], bool f16) {
  if (row_ok && c + 32 <= ncols) {
    const uint4* p = reinterpret_cast<const uint4*>(rowp + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = p[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 t = unpack2(w[k], f16);
        f[q * 8 + 2 * k] = t.x;
        f[q * 8 + 2 * k + 1] = t.y;
      }
    }
  } else {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(rowp);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      f[j] = (row_ok && c + j < ncols) ? unpack2((uint32_t)h[c + j], f16).x : 0.f;
  }
}

// Store 32 packed fp16 (16 words) at rowp[c..c+31], clipped to ncols.
__device__ __forceinline__ void store_row32(__half* rowp, int64_t c, int64_t ncols,
                                            bool row_ok, const uint32_t (&w)[16]) {
  if (!row_ok) return;
  if (c + 32 <= ncols && (reinterpret_cast<uintptr_t>(rowp + c) & 31u) == 0) {
    // Two whole 32-byte sectors per lane, one 256-bit store each.
#pragma unroll
    for (int q = 0; q < 2; ++q) ptx::st_global_v8(rowp + c + 16 * q, w + 8 * q);
  } else if (c + 32 <= ncols) {
    uint4* p = reinterpret_cast<uint4*>(rowp + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  } else {
    uint16_t* h = reinterpret_cast<uint16_t*>(rowp);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c + j < ncols) h[c + j] = (uint16_t)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
  }
}

// Mirror store of a 32x32 fp16 block held one row per lane: lane L writes
// column L of the block as row (c + L) of the destination, columns
// [rbase, rbase+32) clipped to n_lim.  Uses the warp's 32x17-word scratch.
__device__ __forceinline__ void mirror_store32(__half* base, int64_t ld, int64_t c,
                                               int64_t rbase, int64_t n_lim, int lane,
                                               const uint32_t (&w)[16], uint32_t* scratch) {
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
  store_row32(base + dr * ld, rbase, n_lim, dr < n_lim, t);
}

// Per-item view of a launch: the phase, the iteration and the K blocks of an
// item, and that iteration's parameters.
struct ItemInfo {
  int ph, it, kbn;
};

// The items of one persistent processor in the order it runs them: its run
// of the launch's list, or (fused launches) for each iteration k and phase p
// its run of phase p's list.  Every role of the processor (producer, MMA
// issuer, epilogue warps) walks the same sequence.
template <int PHASE>
struct ItemCursor {
  const GemmArgs& a;
  int proc, nproc, k, p, w, w1, step;
  __device__ __forceinline__ ItemCursor(const GemmArgs& a_, int proc_, int nproc_)
      : a(a_), proc(proc_), nproc(nproc_), k(0), p(-1), w(0), w1(0), step(1) {
    if constexpr (PHASE != kPhaseFused) {
      const WorkRange r = work_range(a.starts, proc, nproc, a.n_items);
      w = r.w0;
      w1 = r.w1;
      step = r.step;
    }
  }
  __device__ __forceinline__ bool next(int4& item, ItemInfo& inf) {
    if constexpr (PHASE != kPhaseFused) {
      if (w >= w1) return false;
      item = a.items[w];
      w += step;
      inf = ItemInfo{PHASE, 0, item.w};
      return true;
    } else {
      while (w >= w1) {
        if (++p == 3) {
          p = 0;
          if (++k >= a.n_iters) return false;
        }
        w = w1 = 0;
        if (proc < a.fprocs[p]) {
          const WorkRange r = work_range(a.fstarts[p], proc, a.fprocs[p], a.fn_items[p]);
          w = r.w0;
          w1 = r.w1;
          step = r.step;
        }
      }
      item = a.fitems[p][w];
      w += step;
      inf = ItemInfo{p, k, item.w};
      return true;
    }
  }
};

struct StageParams {
  int src, first;
  float ca, cb, cc;
  bool f16_in, f16_out;  // this iteration's operand format; the Apply output's (the next iteration's)
};
template <int PHASE>
__device__ __forceinline__ StageParams stage_params(const GemmArgs& a, int it) {
  if constexpr (PHASE == kPhaseFused)
    return StageParams{it & 1, it == 0 ? 1 : 0, a.coef[it][0], a.coef[it][1], a.coef[it][2], it < a.f16_iters,
                       it + 1 < a.f16_iters};
  else
    return StageParams{a.src, a.first, a.ca, a.cb, a.cc, a.iter < a.f16_iters, a.iter + 1 < a.f16_iters};
}

// Fused launches: a tile of stage s = 3k + p waits until its matrix's counter
// shows every tile of the stages before it done (`warps` increments per
// tile); the counter never runs ahead of a stage whose tiles are still
// waiting, so reaching the sum over stages < s means all of them finished.
__device__ __forceinline__ uint32_t stage_need(const MatDesc& d, int ph, int it, int warps) {
  return (uint32_t)warps *
         (uint32_t)(it * (2 * d.sym_items + d.apply_items) + (ph >= 1 ? d.sym_items : 0) + (ph >= 2 ? d.sym_items : 0));
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait (same limit and abort protocol as the mbarrier waits) until
// *cnt >= need, then a proxy fence so that the TMA loads issued next see the
// other CTAs' generic stores the counter vouches for.
__device__ __noinline__ bool wait_counter(const int* cnt, int need, volatile int* abort_flag, int* err,
                                          uint64_t limit_ns, int* seen) {
  if ((*seen = ld_acquire(cnt)) < need) {
    const uint64_t t0 = ptx::globaltimer();
    while ((*seen = ld_acquire(cnt)) < need) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(err, 1);
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// An epilogue warp has stored its part of a tile.  The four warps of the CTA
// count themselves on a shared-memory word of the tile's accumulator slot
// (acquire-release at CTA scope, nobody blocks: a warp that gave up on a
// wait never holds the others); the fourth resets the word and, after a
// GPU-scope release fence that covers every store of the tile, adds 1 to the
// matrix's counter.  Called before the warp releases the accumulator, so the
// slot's next tile cannot be counted before the reset.
__device__ __forceinline__ void signal_tile(int* cnt, uint32_t done_word, int lane) {
  __syncwarp();
  if (lane == 0) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(done_word) : "memory");
    if (old == 3) {
      asm volatile("st.relaxed.cta.shared::cta.u32 [%0], 0;" ::"r"(done_word) : "memory");
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      atomicAdd(cnt, 1);
    }
  }
  __syncwarp();
}

// Producer side: a counter value seen before for the same matrix (counters
// only grow) spares the acquire poll.
struct CounterCache {
  int mat = -1, val = 0;
};

template <int PHASE, int MODE, int BN>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, const StageParams& sp, const int4 item,
                                              uint32_t tacc, int quad, int lane, uint32_t* scratch) {
  const MatDesc& d = a.mats[item.x];
  const int64_t m = d.m, n = d.n;
  const int64_t row0 = (int64_t)item.y * kBM;
  const int64_t col0 = (int64_t)item.z * BN;
  const int64_t rbase = row0 + quad * 32;
  const int64_t r = rbase + lane;
  const bool row_ok = r < m;
  const uint32_t tq = tacc + ((uint32_t)(quad * 32) << 16);

  // True scale of the stored iterate: X = xs * X[src] (s/p of the first
  // step's X[0] = p U, else 1/beta' for X stored as beta' X).
  const float bp = a.bvec[item.x];
  const float xs = sp.first ? a.svec[item.x] : 1.f / bp;
  if constexpr (PHASE == kPhaseGram || PHASE == kPhaseGram2) {
    // A tile strictly above the diagonal also writes its transpose (diagonal
    // tiles are computed whole).
    const bool mirror = (int64_t)item.y * kBM / BN < item.z;
    // Gram: A = kappa xs^2 X[src] X[src]^T.  Gram2 with A = kappa X X^T:
    // b A_true + c A_true^2 = (b/kappa) A + (c/kappa^2) A A.
    const float ik = 1.f / d.kappa;
    const float alpha = d.kappa * xs * xs;
    const float gcc = sp.cc * ik * ik, gcb = sp.cb * ik;
    __half* dst = (PHASE == kPhaseGram) ? d.A : d.B;
    const int64_t ld = d.lda;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      const int64_t c = col0 + ch * 32;
      if (c >= m) break;  // warp-uniform
      uint32_t v[32];
      ptx::tmem_ld32(tq + ch * 32, v);
      float f[32];
      if constexpr (PHASE == kPhaseGram) {
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]) * alpha;
      } else {
        float av[32];
        load_row32(d.A + r * ld, c, m, row_ok, av, sp.f16_in);
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = fmaf(gcc, __uint_as_float(v[j]), gcb * av[j]);
        if (a.fold) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (r == c + j) f[j] += sp.ca;
        }
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = pack2(f[2 * k], f[2 * k + 1], sp.f16_in);
      store_row32(dst + r * ld, c, m, row_ok, w);
      if (mirror) mirror_store32(dst, ld, c, rbase, m, lane, w, scratch);
    }
  } else {
    // X' = beta' xs (Z X[src]) stored; the final O = xs (Z X[src]) in fp32.
    const float alpha = MODE == kWriteX ? xs * bp : xs;
    const __half* xsrc = d.X[sp.src];
    __half* xd = d.X[sp.src ^ 1];
    const int64_t ldx = d.ldx;
    const MatPtrs& p = a.ptrs[item.x];
    const float coef = a.lr * d.scale;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      const int64_t c = col0 + ch * 32;
      if (c >= n) break;  // warp-uniform
      uint32_t v[32];
      ptx::tmem_ld32(tq + ch * 32, v);
      float o[32];
      if (a.fold) {  // B already holds a*I: X' = Z X
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = alpha * __uint_as_float(v[j]);
      } else {
        float xv[32];
        load_row32(xsrc + r * ldx, c, n, row_ok, xv, sp.f16_in);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = alpha * fmaf(sp.ca, xv[j], __uint_as_float(v[j]));
      }
      if constexpr (MODE == kWriteX) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = pack2(o[2 * k], o[2 * k + 1], sp.f16_out);
        store_row32(xd + r * ldx, c, n, row_ok, w);
      } else if (row_ok) {
        // All loads of W for this chunk are issued before any store, so the
        // 32 reads are in flight together instead of one round trip each.
        constexpr bool upd = MODE == kUpdateW;
        if (!d.transposed) {
          // W is m x n: row r, columns c..c+31.
          float* wp = p.W + r * d.cols + c;
          if (c + 32 <= n && (d.cols & 3) == 0) {
            float4* w4 = reinterpret_cast<float4*>(wp);
            float4 cur[8];
            if (upd) {
#pragma unroll
              for (int q = 0; q < 8; ++q) cur[q] = __ldcs(w4 + q);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 o4 = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
              if (upd) {
                o4.x = fmaf(a.decay, cur[q].x, -coef * o4.x);
                o4.y = fmaf(a.decay, cur[q].y, -coef * o4.y);
                o4.z = fmaf(a.decay, cur[q].z, -coef * o4.z);
                o4.w = fmaf(a.decay, cur[q].w, -coef * o4.w);
              }
              __stcs(w4 + q, o4);
            }
          } else {
            float cur[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) cur[j] = (upd && c + j < n) ? wp[j] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < n) wp[j] = upd ? fmaf(a.decay, cur[j], -coef * o[j]) : o[j];
          }
        } else {
          // W is n x m: element (c + j, r); lanes hold consecutive r, so
          // each j is one coalesced 128-byte warp access.
          float* wcol = p.W + c * d.cols + r;
          const int64_t ldw = d.cols;
          float cur[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) cur[j] = (upd && c + j < n) ? __ldcs(wcol + j * ldw) : 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c + j < n) __stcs(wcol + j * ldw, upd ? fmaf(a.decay, cur[j], -coef * o[j]) : o[j]);
        }
      }
    }
  }
}

// The epilogue of one item: the launch's own phase, or (fused launches) the
// item's phase and iteration, the last iteration's Apply in the launch's
// final mode.
template <int PHASE, int MODE, int BN>
__device__ __forceinline__ void epilogue_item(const GemmArgs& a, const ItemInfo& inf, const int4 item, uint32_t tacc,
                                              int quad, int lane, uint32_t* scratch) {
  const StageParams sp = stage_params<PHASE>(a, inf.it);
  if constexpr (PHASE != kPhaseFused) {
    epilogue_tile<PHASE, MODE, BN>(a, sp, item, tacc, quad, lane, scratch);
  } else {
    if (inf.ph == kPhaseGram) {
      epilogue_tile<kPhaseGram, kWriteX, BN>(a, sp, item, tacc, quad, lane, scratch);
    } else if (inf.ph == kPhaseGram2) {
      // This epilogue reads A tiles that other CTAs stored: an acquire of the
      // matrix's counter (already past this stage's need, which the producer
      // waited for) orders those stores before this thread's loads.
      (void)ld_acquire(a.counters + item.x);
      epilogue_tile<kPhaseGram2, kWriteX, BN>(a, sp, item, tacc, quad, lane, scratch);
    }
    else if (inf.it < a.n_iters - 1)
      epilogue_tile<kPhaseApply, kWriteX, BN>(a, sp, item, tacc, quad, lane, scratch);
    else if (a.final_mode == kUpdateW)
      epilogue_tile<kPhaseApply, kUpdateW, BN>(a, sp, item, tacc, quad, lane, scratch);
    else
      epilogue_tile<kPhaseApply, kWriteO, BN>(a, sp, item, tacc, quad, lane, scratch);
  }
}

template <int PHASE, int MODE, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = SingleCfg<BN>;
  constexpr int kS = C::kNStages;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve<BN>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns ? a.timeout_ns : kTimeoutNs;

  uint64_t* full = sm.bars;
  uint64_t* empty = sm.bars + kS;
  uint64_t* tfull = sm.bars + 2 * kS;
  uint64_t* tempty = sm.bars + 2 * kS + 2;
  uint64_t* drain = sm.bars + 2 * kS + 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      ptx::mbar_init(ptx::smem_addr(full + s), 1);
      ptx::mbar_init(ptx::smem_addr(empty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(tfull + i), 1);
      ptx::mbar_init(ptx::smem_addr(tempty + i), 4);
    }
    ptx::mbar_init(ptx::smem_addr(drain), 1);
    *sm.abort_flag = 0;
    sm.tile_done[0] = sm.tile_done[1] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(sm.tmem_slot), C::kTmem);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t it = 0;
      bool ok = true;
      ItemCursor<PHASE> cur(a, (int)blockIdx.x, (int)gridDim.x);
      CounterCache cc;
      int4 item;
      ItemInfo inf;
      while (ok && cur.next(item, inf)) {
        const int src = PHASE == kPhaseFused ? (inf.it & 1) : a.src;
        if (PHASE == kPhaseFused) {
          const int need = (int)stage_need(a.mats[item.x], inf.ph, inf.it, 1);
          if (need > 0 && !(cc.mat == item.x && cc.val >= need)) {
            if (!wait_counter(a.counters + item.x, need, sm.abort_flag, a.err, tmo, &cc.val)) { ok = false; break; }
            cc.mat = item.x;
          }
        }
        const CUtensorMap* maps = a.tmaps + (size_t)item.x * kMapsPerMat;
        const CUtensorMap* mapA;
        const CUtensorMap* mapB;
        if (inf.ph == kPhaseGram) {
          mapA = maps + src; mapB = maps + src;
        } else if (inf.ph == kPhaseGram2) {
          mapA = maps + 2; mapB = maps + 2;
        } else {
          mapA = maps + 3; mapB = maps + src;
        }
        const int row0 = item.y * kBM;
        const int col0 = item.z * BN;
        for (int kb = 0; kb < inf.kbn; ++kb, ++it) {
          const uint32_t s = it % kS;
          const uint32_t ph = (it / kS) & 1u;
          if (!wait_bar(ptx::smem_addr(empty + s), ph ^ 1u, sm.abort_flag, a.err, tmo)) { ok = false; break; }
          const uint32_t fb = ptx::smem_addr(full + s);
          ptx::mbar_expect_tx(fb, C::kStageB);
          const uint32_t sa = ptx::smem_addr(sm.stages + s * C::kStageB);
          const uint32_t sb = sa + kABytes;
          const int k0 = kb * kBK;
          ptx::tma_load_2d(sa, mapA, k0, row0, fb);
          ptx::tma_load_2d(sa + kBoxBytes, mapA, k0, row0 + kBox, fb);
#pragma unroll
          for (int q = 0; q < BN / kBox; ++q) {
            if (inf.ph == kPhaseApply)
              ptx::tma_load_2d(sb + q * kBoxBytes, mapB, col0 + q * kBox, k0, fb);
            else
              ptx::tma_load_2d(sb + q * kBoxBytes, mapB, k0, col0 + q * kBox, fb);
          }
        }
      }
      if (!ok || *sm.abort_flag) {
        // Drain: wait (bounded, ignoring the abort flag) for the copies of
        // the last issued stages so none lands after the CTA exits.
        const uint32_t n_out = it < (uint32_t)kS ? it : (uint32_t)kS;
        for (uint32_t i = it - n_out; i < it; ++i)
          wait_slow(ptx::smem_addr(full + (i % kS)), (i / kS) & 1u, sm.abort_flag,
                    a.err, false, kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_sym = ptx::idesc_f16(kBM, BN, 0), idesc_app = ptx::idesc_f16(kBM, BN, 1);
      constexpr uint32_t bdesc_sym = ptx::idesc_bf16(kBM, BN, 0), bdesc_app = ptx::idesc_bf16(kBM, BN, 1);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      bool issued = false;
      ItemCursor<PHASE> cur(a, (int)blockIdx.x, (int)gridDim.x);
      int4 item;
      ItemInfo inf;
      for (; ok && cur.next(item, inf); ++tc) {
        const uint32_t acc = tc & 1u;
        if (!wait_bar(ptx::smem_addr(tempty + acc), ((tc >> 1) & 1u) ^ 1u, sm.abort_flag, a.err, tmo)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + acc * BN;
        const bool mn = inf.ph == kPhaseApply;  // X as the MN-major B operand
        const bool f16 = (PHASE == kPhaseFused ? inf.it : a.iter) < a.f16_iters;
        const uint32_t idesc = f16 ? (mn ? idesc_app : idesc_sym) : (mn ? bdesc_app : bdesc_sym);
        for (int kb = 0; kb < inf.kbn; ++kb, ++it) {
          const uint32_t s = it % kS;
          const uint32_t ph = (it / kS) & 1u;
          if (!wait_bar(ptx::smem_addr(full + s), ph, sm.abort_flag, a.err, tmo)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(sm.stages + s * C::kStageB);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = ptx::desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = mn ? ptx::desc_sw128(sb + kk * 2048, 8192, 1024)
                                   : ptx::desc_sw128(sb + kk * 32, 16, 1024);
            ptx::mma_f16(dt, ad, bd, idesc, (kb | kk) != 0);
          }
          issued = true;
          ptx::mma_commit(ptx::smem_addr(empty + s));
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_addr(tfull + acc));
      }
      if (issued && (!ok || *sm.abort_flag)) {
        ptx::mma_commit(ptx::smem_addr(drain));
        wait_slow(ptx::smem_addr(drain), 0, sm.abort_flag, a.err, false, kDrainTimeoutNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31 for this warp
    uint32_t* scratch = sm.scratch + (warp - 2) * kEpiWords;
    uint32_t tc = 0;
    ItemCursor<PHASE> cur(a, (int)blockIdx.x, (int)gridDim.x);
    int4 item;
    ItemInfo inf;
    for (; cur.next(item, inf); ++tc) {
      const uint32_t acc = tc & 1u;
      if (!wait_bar(ptx::smem_addr(tfull + acc), (tc >> 1) & 1u, sm.abort_flag, a.err, tmo)) break;
      ptx::tc_fence_after();
      epilogue_item<PHASE, MODE, BN>(a, inf, item, tmem_base + acc * BN, quad, lane, scratch);
      if (PHASE == kPhaseFused) signal_tile(a.counters + item.x, ptx::smem_addr(sm.tile_done + acc), lane);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(tempty + acc));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmem);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel (cta_group::2).  A 2-CTA cluster owns one 256x256 output
// tile per work item: rank r holds rows [256*ti + 128*r, +128) of it in its
// TMEM.  Per 64-wide K block each rank loads its 128 rows of A and a 128-row
// half of B into its own shared memory; the transaction bytes of both ranks
// complete on rank 0's `full` barrier, rank 0 issues M=256, N=256 MMAs that
// read both ranks' shared memory, and its commits are multicast to both
// ranks' `empty` (stage free) and `tfull` (accumulator ready) barriers.  Both
// ranks' epilogue warps release an accumulator on rank 0's `tempty` barrier.
// Six 32 KB stages per CTA keep 192 KB of operands in flight per SM.
// ---------------------------------------------------------------------------
struct PairSmem {
  uint8_t* stages;     // kPairStages x (A half 16 KB | B half 16 KB), 1024-aligned
  uint32_t* scratch;   // 4 warps x 32 x 17 words
  uint64_t* bars;      // full[6], empty[6], tfull[2], tempty[2], drain
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  uint32_t* tile_done;  // fused launches: epilogue warps done per accumulator slot
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
  s.tile_done = s.tmem_slot + 2;
  return s;
}

template <int PHASE, int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_pair_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const PairSmem sm = carve_pair(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns ? a.timeout_ns : kTimeoutNs;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

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
    sm.tile_done[0] = sm.tile_done[1] = 0;
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
      ItemCursor<PHASE> cur(a, pair, npairs);
      CounterCache cc;
      int4 item;
      ItemInfo inf;
      while (ok && cur.next(item, inf)) {
        const int src = PHASE == kPhaseFused ? (inf.it & 1) : a.src;
        if (PHASE == kPhaseFused) {  // each rank loads its own halves: both wait
          const int need = (int)stage_need(a.mats[item.x], inf.ph, inf.it, 2);
          if (need > 0 && !(cc.mat == item.x && cc.val >= need)) {
            if (!wait_counter(a.counters + item.x, need, sm.abort_flag, a.err, tmo, &cc.val)) { ok = false; break; }
            cc.mat = item.x;
          }
        }
        const CUtensorMap* maps = a.tmaps + (size_t)item.x * kMapsPerMat;
        const CUtensorMap* mapA;
        const CUtensorMap* mapB;
        if (inf.ph == kPhaseGram) {
          mapA = maps + src; mapB = maps + src;
        } else if (inf.ph == kPhaseGram2) {
          mapA = maps + 2; mapB = maps + 2;
        } else {
          mapA = maps + 3; mapB = maps + src;
        }
        const int rowA = item.y * 256 + (int)rank * 128;
        const int rowB = item.z * 256 + (int)rank * 128;
        for (int kb = 0; kb < inf.kbn; ++kb, ++it) {
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
          if (inf.ph == kPhaseApply) {
            ptx::tma_load_2d_pair(sb, mapB, rowB, k0, fb);
            ptx::tma_load_2d_pair(sb + kBoxBytes, mapB, rowB + kBox, k0, fb);
          } else {
            ptx::tma_load_2d_pair(sb, mapB, k0, rowB, fb);
            ptx::tma_load_2d_pair(sb + kBoxBytes, mapB, k0, rowB + kBox, fb);
          }
        }
      }
      if (leader && (!ok || *sm.abort_flag)) {
        // Drain: the last issued stages' bytes (both ranks') must land before
        // exit; bounded, ignoring the abort flag.
        const uint32_t n_out = it < (uint32_t)kPairStages ? it : (uint32_t)kPairStages;
        for (uint32_t i = it - n_out; i < it; ++i)
          wait_slow(ptx::smem_addr(full + (i % kPairStages)), (i / kPairStages) & 1u, sm.abort_flag,
                    a.err, false, kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_sym = ptx::idesc_f16(256, kBN, 0), idesc_app = ptx::idesc_f16(256, kBN, 1);
      constexpr uint32_t bdesc_sym = ptx::idesc_bf16(256, kBN, 0), bdesc_app = ptx::idesc_bf16(256, kBN, 1);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      bool issued = false;
      ItemCursor<PHASE> cur(a, pair, npairs);
      int4 item;
      ItemInfo inf;
      for (; ok && cur.next(item, inf); ++tc) {
        const uint32_t acc = tc & 1u;
        if (!wait_bar(ptx::smem_addr(tempty + acc), ((tc >> 1) & 1u) ^ 1u, sm.abort_flag, a.err, tmo)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + acc * kBN;
        const bool mn = inf.ph == kPhaseApply;  // X as the MN-major B operand
        const bool f16 = (PHASE == kPhaseFused ? inf.it : a.iter) < a.f16_iters;
        const uint32_t idesc = f16 ? (mn ? idesc_app : idesc_sym) : (mn ? bdesc_app : bdesc_sym);
        for (int kb = 0; kb < inf.kbn; ++kb, ++it) {
          const uint32_t s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1u;
          if (!wait_bar(ptx::smem_addr(full + s), ph, sm.abort_flag, a.err, tmo)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(sm.stages + s * kPairStageBytes);
          const uint32_t sb = sa + kPairHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = ptx::desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = mn ? ptx::desc_sw128(sb + kk * 2048, 8192, 1024)
                                   : ptx::desc_sw128(sb + kk * 32, 16, 1024);
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
    ItemCursor<PHASE> cur(a, pair, npairs);
    int4 item;
    ItemInfo inf;
    for (; cur.next(item, inf); ++tc) {
      const uint32_t acc = tc & 1u;
      if (!wait_bar(ptx::smem_addr(tfull + acc), (tc >> 1) & 1u, sm.abort_flag, a.err, tmo)) break;
      ptx::tc_fence_after();
      item.y = item.y * 2 + (int)rank;  // this rank's 128-row tile
      epilogue_item<PHASE, MODE, kBN>(a, inf, item, tmem_base + acc * kBN, quad, lane, scratch);
      if (PHASE == kPhaseFused) signal_tile(a.counters + item.x, ptx::smem_addr(sm.tile_done + acc), lane);
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

}  // namespace

template <int BN>
cudaError_t configure_bn() {
  constexpr int sm = SingleCfg<BN>::kSmem;
  const cudaFuncAttribute att = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<kPhaseGram, kWriteX, BN>, att, sm)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<kPhaseGram2, kWriteX, BN>, att, sm)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<kPhaseApply, kWriteX, BN>, att, sm)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<kPhaseApply, kUpdateW, BN>, att, sm)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<kPhaseFused, kWriteX, BN>, att, sm)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(ns_gemm_kernel<kPhaseApply, kWriteO, BN>, att, sm);
}

cudaError_t gemm_configure() {
  const cudaError_t e = configure_bn<kBN>();
  return e != cudaSuccess ? e : configure_bn<128>();
}

// Apply launches pick the kernel variant of their final mode, so each
// variant carries only the epilogue it runs.
template <int BN>
cudaError_t launch_bn(int phase, const GemmArgs& a, int grid, cudaStream_t s) {
  constexpr int sm = SingleCfg<BN>::kSmem;
  if (phase == kPhaseFused) {
    ns_gemm_kernel<kPhaseFused, kWriteX, BN><<<grid, kGemmThreads, sm, s>>>(a);
  } else if (phase == kPhaseGram) {
    ns_gemm_kernel<kPhaseGram, kWriteX, BN><<<grid, kGemmThreads, sm, s>>>(a);
  } else if (phase == kPhaseGram2) {
    ns_gemm_kernel<kPhaseGram2, kWriteX, BN><<<grid, kGemmThreads, sm, s>>>(a);
  } else if (a.final_mode == kUpdateW) {
    ns_gemm_kernel<kPhaseApply, kUpdateW, BN><<<grid, kGemmThreads, sm, s>>>(a);
  } else if (a.final_mode == kWriteO) {
    ns_gemm_kernel<kPhaseApply, kWriteO, BN><<<grid, kGemmThreads, sm, s>>>(a);
  } else {
    ns_gemm_kernel<kPhaseApply, kWriteX, BN><<<grid, kGemmThreads, sm, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_gemm(int phase, const GemmArgs& a, int grid, cudaStream_t s, int bn) {
  return bn == 128 ? launch_bn<128>(phase, a, grid, s) : launch_bn<kBN>(phase, a, grid, s);
}

template <int PHASE, int MODE>
cudaError_t configure_pair_one(int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_pair_kernel<PHASE, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  if (e != cudaSuccess || !max_clusters) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, ns_gemm_pair_kernel<PHASE, MODE>, &cfg);
}

cudaError_t gemm_pair_configure(int* max_clusters) {
  cudaError_t e;
  if ((e = configure_pair_one<kPhaseGram, kWriteX>(max_clusters)) != cudaSuccess) return e;
  if ((e = configure_pair_one<kPhaseGram2, kWriteX>(nullptr)) != cudaSuccess) return e;
  if ((e = configure_pair_one<kPhaseApply, kWriteX>(nullptr)) != cudaSuccess) return e;
  if ((e = configure_pair_one<kPhaseApply, kUpdateW>(nullptr)) != cudaSuccess) return e;
  if ((e = configure_pair_one<kPhaseFused, kWriteX>(nullptr)) != cudaSuccess) return e;
  return configure_pair_one<kPhaseApply, kWriteO>(nullptr);
}

template <int PHASE, int MODE>
cudaError_t launch_pair_one(const GemmArgs& a, int clusters, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel<PHASE, MODE>, a);
}

cudaError_t launch_gemm_pair(int phase, const GemmArgs& a, int clusters, cudaStream_t s) {
  if (phase == kPhaseFused) return launch_pair_one<kPhaseFused, kWriteX>(a, clusters, s);
  if (phase == kPhaseGram) return launch_pair_one<kPhaseGram, kWriteX>(a, clusters, s);
  if (phase == kPhaseGram2) return launch_pair_one<kPhaseGram2, kWriteX>(a, clusters, s);
  if (a.final_mode == kUpdateW) return launch_pair_one<kPhaseApply, kUpdateW>(a, clusters, s);
  if (a.final_mode == kWriteO) return launch_pair_one<kPhaseApply, kWriteO>(a, clusters, s);
  return launch_pair_one<kPhaseApply, kWriteX>(a, clusters, s);
}

}  // namespace dmuon
