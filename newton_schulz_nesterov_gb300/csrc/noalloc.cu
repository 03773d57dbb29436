// dmuon_newton_schulz_noalloc: standalone Newton-Schulz of one matrix that
// allocates no device memory.
//
// For callers that cannot call cudaMalloc: code that runs inside a host
// framework whose allocator owns all device memory and forbids side
// allocations, plugins that are handed only input and output buffers, and
// latency-critical paths that cannot afford cudaMalloc's implicit device
// synchronisation.  Everything the computation needs beyond its input and
// output -- the fp16 iterate X (ping/pong), the products A and B, the
// per-tile sums of squares and maxima, the matrix descriptor, four TMA
// tensor maps and the work lists -- lives in one file-scope static
// __device__ array of kNaScratchBytes (about 13.1 MB).  Every GPU that loads
// the library holds that array until the process exits.
//
// Limits: short side min(rows, cols) <= 1024 and rows*cols <= 2^21; larger
// matrices are rejected with DMUON_ERR_ARG before anything is launched.
//
// The array is shared by every call and keeps the last call's contents.
// Each call clears what must start at zero (the non-finite flag, the
// wait-timeout word, the redo flag) and overwrites everything else it reads.
// Calls whose GPU work overlaps (different streams without ordering, or
// several host threads) race on the array and give wrong results.
//
// Set-up: the first call on a device (with that device current) resolves the
// array's device address with cudaGetSymbolAddress, raises the kernels'
// shared-memory limit and reads the SM count; later calls on that device
// reuse the cached values.  A set-up that fails for a reason other than an
// unsupported device is tried again by the next call.
//
// Every call copies its descriptor, tensor maps and work lists from a host
// staging image with cudaMemcpyAsync, so a call cannot be recorded into a
// CUDA graph: while `stream` is being captured the entry point returns
// DMUON_ERR_ARG without touching the device.
//
// Arithmetic: the same kernels as dmuon_newton_schulz on single CTAs with
// the unfolded epilogue (the Z product writes b A + c A A, the X product
// adds a X read from X), so roundings differ from dmuon_newton_schulz's.
// Each call starts from the prescale p = 1 for X0 = p U; inputs whose
// entries are far from 1 take the redo pass (one more read of the input).
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/dmuon.h"
#include "coeffs.cuh"
#include "common.cuh"

namespace dmuon {
namespace {

constexpr int64_t kNaMaxShort = 1024;
constexpr int64_t kNaMaxElems = int64_t(1) << 21;
// X rows are padded to a multiple of 8 elements: at most 7 extra per row.
constexpr int64_t kNaXElems = kNaMaxElems + 8 * kNaMaxShort;
constexpr int64_t kNaMaxTiles = 40960;        // >= ceil(r/64)*ceil(c/64) within the limits
constexpr int64_t kNaMaxSymItems = 20;        // short side <= 1024: 10 super-tiles x 2
constexpr int64_t kNaMaxApplyItems = 8448;    // >= ceil(m/128)*ceil(n/256) within the limits

constexpr size_t na_round(size_t b) { return (b + 255) & ~size_t(255); }
constexpr size_t kOffX0 = 0;
constexpr size_t kOffX1 = kOffX0 + na_round(kNaXElems * 2);
constexpr size_t kOffA = kOffX1 + na_round(kNaXElems * 2);
constexpr size_t kOffB = kOffA + na_round(kNaMaxShort * kNaMaxShort * 2);
constexpr size_t kOffPartials = kOffB + na_round(kNaMaxShort * kNaMaxShort * 2);
constexpr size_t kOffTmax = kOffPartials + na_round(kNaMaxTiles * 4);
constexpr size_t kOffMaps = kOffTmax + na_round(kNaMaxTiles * 4);
constexpr size_t kOffDesc = kOffMaps + na_round(kMapsPerMat * sizeof(CUtensorMap));
constexpr size_t kOffPtrs = kOffDesc + na_round(sizeof(MatDesc));
constexpr size_t kOffPrefix = kOffPtrs + na_round(sizeof(MatPtrs));
constexpr size_t kOffWords = kOffPrefix + na_round(2 * sizeof(int64_t));  // s/p, flag, err, p, redo, beta'
constexpr size_t kOffItems0 = kOffWords + 256;
constexpr size_t kOffItems1 = kOffItems0 + na_round(kNaMaxSymItems * 16);
constexpr size_t kOffItems2 = kOffItems1 + na_round(kNaMaxSymItems * 16);
constexpr size_t kNaScratchBytes = kOffItems2 + na_round(kNaMaxApplyItems * 16);

// The scratch of every dmuon_newton_schulz_noalloc call.  In host code this
// name is only a stand-in; the device address comes from
// cudaGetSymbolAddress in na_setup().
static __device__ __align__(256) unsigned char g_na_scratch[kNaScratchBytes];

// Staging image of everything the host writes into the scratch per call;
// laid out to be copied with one cudaMemcpyAsync to kOffMaps.
struct alignas(256) HostImage {
  CUtensorMap maps[kMapsPerMat];
  alignas(256) MatDesc desc;
  alignas(256) MatPtrs ptrs;
  alignas(256) int64_t prefix[2];
  alignas(256) uint32_t words[64];  // [0] s/p, [1] flag, [2] err, [3] p (float bits), [4] redo, [5] beta'
  alignas(256) int4 items0[kNaMaxSymItems];
  alignas(256) int4 items1[kNaMaxSymItems];
  alignas(256) int4 items2[kNaMaxApplyItems];
};
static_assert(offsetof(HostImage, desc) == kOffDesc - kOffMaps, "image layout");
static_assert(offsetof(HostImage, ptrs) == kOffPtrs - kOffMaps, "image layout");
static_assert(offsetof(HostImage, prefix) == kOffPrefix - kOffMaps, "image layout");
static_assert(offsetof(HostImage, words) == kOffWords - kOffMaps, "image layout");
static_assert(offsetof(HostImage, items0) == kOffItems0 - kOffMaps, "image layout");
static_assert(offsetof(HostImage, items1) == kOffItems1 - kOffMaps, "image layout");
static_assert(offsetof(HostImage, items2) == kOffItems2 - kOffMaps, "image layout");

struct DeviceSetup {
  bool done = false;
  int rc = DMUON_OK;
  unsigned char* base = nullptr;
  int num_sms = 0;
};

constexpr int kNaMaxDevices = 64;
std::mutex g_na_mutex;
DeviceSetup g_na_dev[kNaMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// Once per device, with that device current.
int na_setup(int dev, DeviceSetup** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return DMUON_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  DeviceSetup& s = g_na_dev[dev];
  if (!s.done) {
    s.rc = DMUON_OK;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    void* p = nullptr;
    if (major != 10 || minor != 3) {
      s.rc = DMUON_ERR_UNSUPPORTED;
    } else if (cudaGetSymbolAddress(&p, g_na_scratch) != cudaSuccess || p == nullptr) {
      s.rc = DMUON_ERR_CUDA;
    } else if (gemm_configure() != cudaSuccess) {
      s.rc = DMUON_ERR_CUDA;
    } else {
      s.base = static_cast<unsigned char*>(p);
      if (!g_na_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
          g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
      if (!g_na_encode) s.rc = DMUON_ERR_CUDA;
    }
    if (s.rc != DMUON_OK) cudaGetLastError();
    // Only an unsupported device is final; other failures are retried.
    s.done = s.rc == DMUON_OK || s.rc == DMUON_ERR_UNSUPPORTED;
  }
  *out = &s;
  return s.rc;
}

bool na_encode(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)kBox, (cuuint32_t)kBox};
  cuuint32_t estr[2] = {1, 1};
  return g_na_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int64_t na_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" int dmuon_newton_schulz_noalloc(const float* input, float* output, int64_t rows,
                                           int64_t cols, int ns_steps, const float* coeffs,
                                           float eps, int sync_status, void* stream_) {
  // ---- host checks, before anything touches the device
  if (!input || !output) return DMUON_ERR_ARG;
  if (((uintptr_t)input & 15u) || ((uintptr_t)output & 15u)) return DMUON_ERR_ALIGN;
  if (rows <= 0 || cols <= 0) return DMUON_ERR_ARG;
  const int64_t m = std::min(rows, cols), n = std::max(rows, cols);
  if (m > kNaMaxShort || rows * cols > kNaMaxElems) return DMUON_ERR_ARG;
  const uintptr_t ib = (uintptr_t)input, ob = (uintptr_t)output, bytes = (uintptr_t)(rows * cols * 4);
  if (ib < ob + bytes && ob < ib + bytes) return DMUON_ERR_ARG;  // overlap
  if (ns_steps < 0 || ns_steps > DMUON_MAX_NS_STEPS) return DMUON_ERR_ARG;
  if (coeffs)
    for (int i = 0; i < 3 * ns_steps; ++i)
      if (!std::isfinite(coeffs[i])) return DMUON_ERR_ARG;
  if (!std::isfinite(eps)) return DMUON_ERR_ARG;
  if (eps <= 0.f) eps = 1e-7f;
  if (!direct_table_fits(ns_steps, coeffs, nullptr, 0)) return DMUON_ERR_ARG;  // fp16 range
  cudaStream_t stream = (cudaStream_t)stream_;
  {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) { cudaGetLastError(); return DMUON_ERR_CUDA; }
    if (cap != cudaStreamCaptureStatusNone) return DMUON_ERR_ARG;  // see the top of this file
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return DMUON_ERR_CUDA; }
  DeviceSetup* ds = nullptr;
  if (int rc = na_setup(dev, &ds)) return rc;
  unsigned char* base = ds->base;

  // ---- descriptor, tensor maps and work lists of this matrix
  static thread_local HostImage img;
  std::memset(&img.desc, 0, sizeof img.desc);
  MatDesc& d = img.desc;
  d.rows = rows;
  d.cols = cols;
  d.transposed = rows > cols ? 1 : 0;
  d.m = m;
  d.n = n;
  d.ldx = (n + 7) / 8 * 8;
  d.lda = (m + 7) / 8 * 8;
  d.X[0] = reinterpret_cast<__half*>(base + kOffX0);
  d.X[1] = reinterpret_cast<__half*>(base + kOffX1);
  d.A = reinterpret_cast<__half*>(base + kOffA);
  d.B = reinterpret_cast<__half*>(base + kOffB);
  d.tile0 = 0;
  d.tiles_c = (int32_t)na_cdiv(cols, kMomTile);
  d.scale = 1.f;
  d.kappa = scale_kappa(m);
  d.beta = scale_beta(n);
  const int64_t n_tiles = na_cdiv(rows, kMomTile) * d.tiles_c;
  if (n_tiles > kNaMaxTiles || na_cdiv(m, kBM) * na_cdiv(n, kBN) > kNaMaxApplyItems) return DMUON_ERR_ARG;
  img.ptrs = MatPtrs{output, input, nullptr, nullptr};
  img.prefix[0] = 0;
  img.prefix[1] = n_tiles;
  std::memset(img.words, 0, sizeof img.words);
  const float p_start = 1.f;
  std::memcpy(&img.words[3], &p_start, 4);
  if (!na_encode(&img.maps[0], d.X[0], m, n, d.ldx) || !na_encode(&img.maps[1], d.X[1], m, n, d.ldx) ||
      !na_encode(&img.maps[2], d.A, m, m, d.lda) || !na_encode(&img.maps[3], d.B, m, m, d.lda))
    return DMUON_ERR_CUDA;
  int n_sym = 0, n_apply = 0;
  const int64_t T = na_cdiv(m, 256);
  const int kg = (int)na_cdiv(n, kBK), km = (int)na_cdiv(m, kBK);
  for (int64_t I = 0; I < T; ++I)
    for (int64_t J = I; J < T; ++J)
      for (int h = 0; h < 2; ++h) {
        const int64_t ti = 2 * I + h;
        if (ti * kBM >= m) continue;
        img.items0[n_sym] = make_int4(0, (int)ti, (int)J, kg);
        img.items1[n_sym] = make_int4(0, (int)ti, (int)J, km);
        ++n_sym;
      }
  for (int64_t ti = 0; ti < na_cdiv(m, kBM); ++ti)
    for (int64_t tj = 0; tj < na_cdiv(n, kBN); ++tj) img.items2[n_apply++] = make_int4(0, (int)ti, (int)tj, km);

  // One copy of the image (pageable source: staged before return), which
  // also zeroes the flag, timeout and redo words and sets p = 1.
  const size_t img_bytes = offsetof(HostImage, items2) + sizeof(int4) * (size_t)n_apply;
  cudaError_t e = cudaMemcpyAsync(base + kOffMaps, &img, img_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return DMUON_ERR_CUDA;

  const MatDesc* dd = reinterpret_cast<const MatDesc*>(base + kOffDesc);
  const MatPtrs* dp = reinterpret_cast<const MatPtrs*>(base + kOffPtrs);
  const int64_t* dprefix = reinterpret_cast<const int64_t*>(base + kOffPrefix);
  float* svec = reinterpret_cast<float*>(base + kOffWords);
  int* flags = reinterpret_cast<int*>(base + kOffWords + 4);
  int* err = reinterpret_cast<int*>(base + kOffWords + 8);
  float* pscale = reinterpret_cast<float*>(base + kOffWords + 12);
  int* redo = reinterpret_cast<int*>(base + kOffWords + 16);
  float* bvec = reinterpret_cast<float*>(base + kOffWords + 20);
  float* partials = reinterpret_cast<float*>(base + kOffPartials);
  float* tmax = reinterpret_cast<float*>(base + kOffTmax);
  const CUtensorMap* maps = reinterpret_cast<const CUtensorMap*>(base + kOffMaps);

  const int grid_e = (int)std::min<int64_t>(n_tiles, (int64_t)ds->num_sms * 8);
  const int grid_m = (int)std::min<int64_t>(n_tiles, (int64_t)ds->num_sms * kMomCtasPerSm);
  for (int pass = 0; pass < 2; ++pass) {  // momentum-free pass, then the redo pass if p missed
    if (launch_mom(MomArgs{dd, dp, dprefix, 1, n_tiles, 0.f, 0, 1, partials, tmax, pscale, redo, pass}, grid_m,
                   stream) != cudaSuccess)
      return DMUON_ERR_CUDA;
    if (launch_finalize(FinalizeArgs{dd, dprefix, partials, tmax, 1, eps, svec, bvec, pscale, redo, flags, pass},
                        stream) != cudaSuccess)
      return DMUON_ERR_CUDA;
  }
  if (ns_steps == 0) {
    if (launch_update0(Update0Args{dd, dp, dprefix, 1, n_tiles, svec, 0.f, 1.f, 1}, grid_e, stream) != cudaSuccess)
      return DMUON_ERR_CUDA;
  }
  const int4* items[3] = {reinterpret_cast<const int4*>(base + kOffItems0),
                          reinterpret_cast<const int4*>(base + kOffItems1),
                          reinterpret_cast<const int4*>(base + kOffItems2)};
  const int counts[3] = {n_sym, n_sym, n_apply};
  for (int k = 0; k < ns_steps; ++k) {
    const float* row = coefficient_row(coeffs, k);  // NULL: YOU_COEFFICIENTS
    for (int p = 0; p < 3; ++p) {
      GemmArgs a{};
      a.mats = dd;
      a.ptrs = dp;
      a.tmaps = maps;
      a.items = items[p];
      a.n_items = counts[p];
      a.src = k & 1;
      a.ca = row[0];
      a.cb = row[1];
      a.cc = row[2];
      a.first = k == 0;
      a.iter = k;
      a.f16_iters = 1 << 30;  // fp16 operands in every iteration
      a.final_mode = (k == ns_steps - 1) ? kWriteO : kWriteX;
      a.lr = 0.f;
      a.decay = 1.f;
      a.svec = svec;
      a.bvec = bvec;
      a.err = err;
      const int grid = std::min(counts[p], ds->num_sms);
      if (launch_gemm(p, a, grid, stream) != cudaSuccess) return DMUON_ERR_CUDA;
    }
  }
  if (!sync_status) return DMUON_OK;
  // Synchronous mode: wait, then report what the kernels recorded.
  int words[3] = {0, 0, 0};
  if (cudaMemcpyAsync(words, base + kOffWords, sizeof words, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  if (words[2]) return DMUON_ERR_TIMEOUT;
  if (words[1]) return DMUON_ERR_NONFINITE;
  return DMUON_OK;
}
