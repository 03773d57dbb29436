/*
 * dmuon.h -- C ABI of the GB300 (sm_103a) owner-side Muon step.
 *
 * One call runs, for every matrix of a packed list of mixed-shape fp32
 * matrices, the step that the owner rank of a Muon-target weight performs
 * (DMuon "HSDP Training", section "What Happens Under the Hood": the owner
 * runs momentum, Newton-Schulz, weight decay and the update):
 *
 *   M <- mu*M + G                                  (momentum, fp32)
 *   U  = G + mu*M   (nesterov=1)   or   U = M      (Nesterov input)
 *   Y  = U^T if rows > cols else U                 (orientation rule)
 *   X  = Y / (||Y||_F + eps)                       (Frobenius normalisation)
 *   repeat ns_steps times with per-step (a,b,c):   (quintic Newton-Schulz)
 *       A = X X^T;  B = b*A + c*A*A;  X = a*X + B*X
 *   O  = X^T if transposed else X
 *   W <- (1 - lr*wd)*W - lr*scale(rows,cols)*O     (decoupled decay + update)
 *
 * Passages: DMuon "API Reference", section "Muon" (signature defaults
 * lr=0.02, momentum=0.95, weight_decay=0.0, ns_steps=5, nesterov=True; the
 * nesterov argument's note on the lookahead input); section
 * "direct_newton_schulz" (the recurrence, eps=1e-7, coefficient list length
 * = iteration count); section "gram_newton_schulz_factors" (normaliser
 * = norm + eps under the orientation rule); section "YOU_COEFFICIENTS" (the
 * default five-row table used here).
 *
 * Precision: momentum and the update are fp32; the Newton-Schulz products
 * run on 16-bit tensor cores with fp32 accumulation, with X, A, B held in 16
 * bits between products, each with a power-of-two scale that keeps it in
 * fp16's normal range (X0 = p U with p chosen from max |U|; later X as
 * beta X, beta ~ sqrt(n); A as kappa X X^T, kappa ~ m).  The first
 * iterations use fp16 operands, whose three extra mantissa bits over bf16
 * cut the rounding error about eightfold where it matters most (small
 * singular values are still in their linear regime); the direct backend's
 * later iterations use bf16, which costs less energy at the same rate
 * (dmuon_set_fp16_iterations; the Gram backend, the small-matrix kernel and
 * the allocation-free entry point are fp16 throughout).  The last
 * iteration's output goes to the update in fp32.  Coefficient tables that
 * could drive a buffer past the fp16 range for some input are refused
 * (DMUON_ERR_ARG).
 *
 * Threading/streams: a handle is not thread-safe.  Calls on one handle are
 * asynchronous on the given stream and must be issued on one stream (or be
 * ordered by the caller), because they share the handle's workspace.
 *
 * Return codes: 0 on success, a negative DMUON_ERR_* otherwise.  Every
 * argument check happens on the host before anything is launched, so an
 * error return means no kernel of that call ran.
 */
#ifndef DMUON_H
#define DMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DMUON_OK               0
#define DMUON_ERR_ARG         -1  /* null pointer, bad size, bad option      */
#define DMUON_ERR_ALIGN       -2  /* a matrix pointer is not 16-byte aligned  */
#define DMUON_ERR_OOM         -3  /* workspace allocation failed              */
#define DMUON_ERR_CUDA        -4  /* a CUDA runtime/driver call failed        */
#define DMUON_ERR_NONFINITE   -5  /* an input matrix held Inf/NaN             */
#define DMUON_ERR_TIMEOUT     -6  /* a kernel's bounded wait ran out          */
#define DMUON_ERR_UNSUPPORTED -7  /* device is not compute capability 10.3    */

/* Largest accepted sizes: any side up to 2^20, short side up to 32768. */
#define DMUON_MAX_DIM        (1 << 20)
#define DMUON_MAX_SHORT_SIDE 32768
#define DMUON_MAX_NS_STEPS   64

/* Shape of one weight matrix: rows x cols, fp32, contiguous row-major
 * (the layout of a PyTorch nn.Linear weight, [out_features, in_features]). */
typedef struct {
    int64_t rows;
    int64_t cols;
} dmuon_shape_t;

/* Newton-Schulz backends (DMuon "API Reference", section "NewtonSchulz",
 * argument backend).  DIRECT iterates on the m x n matrix (section
 * "direct_newton_schulz"); GRAM iterates on its m x m Gram matrix with
 * restarts (section "gram_newton_schulz"): per restart window
 * R = X X^T, then per step Z = a I + b R + c R^2, Q <- Z Q, R <- Z R Z, and
 * X <- Q X at each restart and at the end.  Same function in exact
 * arithmetic; GRAM needs 3 m^2 n + 7 m^3 multiply-adds for five steps with
 * one restart against 7.5 m^2 n + 2.5 m^3 for DIRECT (symmetric products
 * count half), so it is cheaper whenever n > m.  GRAM keeps R and R Z in
 * fp16 scaled by a power of two near m (at most 1024), Z and Q in fp16, and
 * restarts explicitly (X <- Q X, a new R from X); it never runs a window
 * longer than two steps (a longer one is split, which leaves the result
 * unchanged in exact arithmetic: the window products R Z and Z Q, symmetric
 * only in exact arithmetic, are stored symmetric in fp16, and over three or
 * more steps that costs accuracy on inputs with widely spread singular
 * values).  Its default
 * coefficients are the Polar Express table ("API Reference", sections
 * "gram_newton_schulz" and "POLAR_EXPRESS_COEFFICIENTS";
 * dmuon_polar_express_coefficients(ns_steps, 1e-3, 1, 1.05)).  Matrices
 * taken by the small-matrix kernel (dmuon_set_small_path) run the direct
 * iteration with the same table either way. */
#define DMUON_BACKEND_DIRECT 0
#define DMUON_BACKEND_GRAM   1

/* Options of a step; dmuon_default_opts() fills the defaults. */
typedef struct {
    float weight_decay;   /* Muon weight decay; default 0.0                */
    float eps;            /* normalisation epsilon; default 1e-7           */
    int   nesterov;       /* 1 = Nesterov lookahead input (default), 0 = M */
    int   scale_mode;     /* update scale: 0 = sqrt(max(1, rows/cols))
                           * (default), 1 = 1, 2 = 0.2*sqrt(max(rows,cols)) */
    const float* coeffs;  /* NULL: DIRECT the YOU_COEFFICIENTS rows, last
                           * row repeated past five steps; GRAM the Polar
                           * Express rows; else host memory of ns_steps
                           * rows of (a, b, c), row-major                  */
    int   backend;        /* DMUON_BACKEND_DIRECT (default) or _GRAM       */
    const int* restarts;  /* GRAM: restart positions (host), a position k
                           * starting a new window before step k (0-based);
                           * positions outside (0, ns_steps) are ignored.
                           * NULL = the pages' default {2}                  */
    int   n_restarts;     /* entries of restarts (0..DMUON_MAX_NS_STEPS)   */
} dmuon_opts_t;

/* Opaque handle: owns the workspace, the plan cache and the status flags. */
typedef struct dmuon_ctx* dmuon_handle_t;

/* Fill *opts with the defaults (weight_decay 0, eps 1e-7, nesterov 1,
 * scale_mode 0, coeffs NULL, backend DIRECT, restarts NULL).  No-op on
 * NULL.  The pages' own default backend is GRAM; DIRECT is the default
 * here because it is the iteration the step is specified by. */
void dmuon_default_opts(dmuon_opts_t* opts);

/* Create a handle on CUDA device `device` (which becomes current for the
 * calling thread).  Returns DMUON_ERR_UNSUPPORTED unless the device has
 * compute capability 10.3.  *out is set to NULL on failure. */
int dmuon_create(dmuon_handle_t* out, int device);

/* Free the handle and its workspace (synchronises the device first).
 * NULL is a no-op. */
void dmuon_destroy(dmuon_handle_t h);

/* Bytes of device memory a step over `shapes` allocates with the default
 * chunking (fp16 X ping/pong, A and B for the largest chunk, plus small
 * per-matrix arrays), for either tiling.  Host only. */
int dmuon_workspace_bytes(const dmuon_shape_t* shapes, int n_mats,
                          size_t* out_bytes);

/* As dmuon_workspace_bytes for a backend: DMUON_BACKEND_GRAM plans hold
 * X ping/pong plus eight m x m fp16 buffers per matrix of the largest
 * chunk.  DMUON_ERR_ARG for an unknown backend.  Host only. */
int dmuon_workspace_bytes_ex(const dmuon_shape_t* shapes, int n_mats, int backend, size_t* out_bytes);

/*
 * One owner-side Muon step over n_mats matrices (see the top of this file).
 *
 *   params[i]   device, fp32 rows_i x cols_i, updated in place   (W)
 *   grads[i]    device, fp32 rows_i x cols_i, read only          (G)
 *   momentum[i] device, fp32 rows_i x cols_i, updated in place   (M)
 *   shapes[i]   host
 *   params, grads, momentum, shapes: host arrays of n_mats entries.
 *   lr, mu      Muon learning rate and momentum coefficient.
 *   ns_steps    number of Newton-Schulz iterations, 0..DMUON_MAX_NS_STEPS.
 *   opts        NULL = defaults.  backend DMUON_BACKEND_GRAM selects the
 *               Gram-space iteration (see dmuon_gram_newton_schulz;
 *               DMUON_ERR_UNSUPPORTED without 2-CTA clusters).  Either
 *               backend returns DMUON_ERR_ARG for a coefficient table that
 *               could drive an fp16 buffer past its range for some input
 *               (dmuon_last_error says which step and buffer).
 *   stream      a cudaStream_t (NULL = legacy default stream).
 *
 * The caller owns all matrix memory; pointers must be 16-byte aligned and
 * the three matrices of one entry must not overlap.  n_mats == 0 returns
 * DMUON_OK without launching.  The first call with a new shape list plans
 * and allocates the workspace (synchronous); later calls with the same
 * shapes only launch.  Asynchronous: completion and non-finite detection
 * are observed through dmuon_get_status().
 *
 * CUDA graphs: while `stream` is being captured the call only records its
 * kernel launches; the plan, the update scales and the pointer set must
 * already exist from an earlier uncaptured call with the same shapes,
 * scale_mode and buffers, else DMUON_ERR_ARG.  lr, mu, the coefficients and
 * the other scalars are recorded by value in the graph.
 */
int dmuon_step(dmuon_handle_t h, float* const* params,
               const float* const* grads, float* const* momentum,
               const dmuon_shape_t* shapes, int n_mats, float lr, float mu,
               int ns_steps, const dmuon_opts_t* opts, void* stream);

/*
 * Standalone Newton-Schulz orthogonalisation (DMuon "API Reference",
 * section "direct_newton_schulz"): outputs[i] = O of inputs[i], same shape,
 * fp32.  inputs[i] and outputs[i] are device fp32 rows_i x cols_i,
 * 16-byte aligned, and may not overlap.  coeffs: NULL = default table as in
 * dmuon_opts_t, else ns_steps host rows of (a,b,c); DMUON_ERR_ARG for a table
 * outside the fp16 range as in dmuon_step.  eps <= 0 selects 1e-7.
 */
int dmuon_newton_schulz(dmuon_handle_t h, const float* const* inputs,
                        float* const* outputs, const dmuon_shape_t* shapes,
                        int n_mats, int ns_steps, const float* coeffs,
                        float eps, void* stream);

/*
 * Standalone Newton-Schulz with the Gram-space backend (DMuon "API
 * Reference", section "gram_newton_schulz"): as dmuon_newton_schulz, with
 * restart positions `restarts` (host, n_restarts entries; NULL = {2}; a
 * window longer than two steps is split) and coeffs NULL = the Polar
 * Express table.  DMUON_ERR_ARG if the coefficient table could drive a
 * Gram-space buffer past the fp16 range for some input
 * (dmuon_gram_check_coefficients, which also says why);
 * DMUON_ERR_UNSUPPORTED without 2-CTA clusters.
 */
int dmuon_gram_newton_schulz(dmuon_handle_t h, const float* const* inputs,
                             float* const* outputs, const dmuon_shape_t* shapes,
                             int n_mats, int ns_steps, const float* coeffs,
                             const int* restarts, int n_restarts, float eps,
                             void* stream);

/*
 * AdamW on a list of flat fp32 tensors, in place (the non-Muon half of
 * Muon.step: DMuon "API Reference", section "Muon", defaults adamw_lr 1e-3,
 * adamw_betas (0.9, 0.999), adamw_weight_decay 0.01, adamw_eps 1e-8).
 * Decoupled decay and bias correction, as PyTorch's AdamW:
 *   p *= 1 - lr*wd;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr/(1-b1^step) * m / (sqrt(v)/sqrt(1-b2^step) + eps)
 * params, grads, exp_avg, exp_avg_sq: host arrays of n device pointers to
 * numels[i] fp32 elements (4-byte aligned; 16-byte aligned with numel % 4 ==
 * 0 takes the vector path), pairwise distinct.  step >= 1 is the step count
 * after this update; 0 <= beta < 1.  Asynchronous on `stream`.
 */
int dmuon_adamw_step(dmuon_handle_t h, float* const* params,
                     const float* const* grads, float* const* exp_avg,
                     float* const* exp_avg_sq, const int64_t* numels, int n,
                     float lr, float beta1, float beta2, float eps,
                     float weight_decay, int step, void* stream);

/*
 * Segmented gradient-norm clipping (DMuon "API Reference", sections
 * "clip_grad_norm_" and "clip_grad_norm_buckets_"): for every bucket b,
 * norm_b = ||concatenation of its gradients||_2 (fixed-order fp64 sum of
 * fixed-order fp32 tile sums), coef_b = max_norm / (norm_b + 1e-6), and its
 * gradients are scaled by coef_b in place when coef_b < 1.
 *   grads[i]  device fp32, numels[i] elements, 4-byte aligned
 *   buckets   host, n bucket indices in [0, n_buckets); NULL = one bucket
 *   max_norm  <= 0: statistics only (no scaling; coef reported as -1)
 *   norms_out, coefs_out  host, n_buckets floats each, or NULL.  When either
 *             is given the call waits for the stream and fills them; a
 *             non-finite norm reports an Inf/NaN gradient (found_inf).
 */
int dmuon_clip_grad_norm(dmuon_handle_t h, float* const* grads,
                         const int64_t* numels, int n, const int* buckets,
                         int n_buckets, float max_norm, float* norms_out,
                         float* coefs_out, void* stream);

/*
 * Allocation-free standalone Newton-Schulz of ONE matrix.  The pages have no
 * counterpart of this entry point; it exists for callers that may not call
 * cudaMalloc (a host framework whose allocator owns all device memory, a
 * plugin that is handed only its input and output buffers, a latency path
 * that cannot take cudaMalloc's implicit synchronisation).  It needs no
 * handle and allocates nothing: its scratch (fp16 iterate, products, tile
 * sums and maxima, descriptor, tensor maps, work lists) is one file-scope
 * static device array of about 13.1 MB that every GPU loading the library
 * holds until process exit.
 *
 *   input, output  device fp32 rows x cols, row-major, 16-byte aligned, not
 *                  overlapping; output = O of input (the same maths as
 *                  dmuon_newton_schulz on single-CTA kernels with the
 *                  unfolded epilogue -- Z written as b A + c A A, a X added
 *                  from X -- so roundings differ from dmuon_newton_schulz's)
 *   limits         min(rows, cols) <= 1024 and rows*cols <= 2^21, else
 *                  DMUON_ERR_ARG before anything is launched
 *   ns_steps, coeffs, eps   as in dmuon_newton_schulz
 *   sync_status    0: asynchronous on `stream`, device-side problems are not
 *                  reported; non-zero: the call waits for its work and
 *                  returns DMUON_ERR_NONFINITE / DMUON_ERR_TIMEOUT if the
 *                  kernels recorded one
 *   stream         a cudaStream_t on the current device
 *
 * The first call on a device does a one-time set-up with that device current
 * (cudaGetSymbolAddress of the array, kernel attributes); a set-up that
 * failed for any reason but an unsupported device is retried by the next
 * call.  Each call uploads its descriptor, maps and work lists with
 * cudaMemcpyAsync from host memory, so it cannot be recorded into a CUDA
 * graph: while `stream` is being captured it returns DMUON_ERR_ARG and
 * touches nothing.  Every call shares the array and leaves its contents
 * behind; each call zeroes what must start at zero.  Calls whose GPU work
 * overlaps in time (unordered streams, several host threads) race on the
 * array.
 */
int dmuon_newton_schulz_noalloc(const float* input, float* output,
                                int64_t rows, int64_t cols, int ns_steps,
                                const float* coeffs, float eps,
                                int sync_status, void* stream);

/*
 * Wait for the handle's stream work to finish and report what the kernels
 * recorded since the previous call of this function: per-matrix flags of
 * the last planned list (bit 0: non-finite input) are copied to
 * flags[0..min(n_flags, n_mats)) when flags != NULL, then cleared.
 * Returns DMUON_ERR_TIMEOUT if a kernel's bounded wait ran out,
 * DMUON_ERR_NONFINITE if any flag is set, DMUON_OK otherwise.
 */
int dmuon_get_status(dmuon_handle_t h, int* flags, int n_flags);

/* Text describing the most recent failure on this handle (which call or
 * CUDA error), "" if none; valid until the next call on the handle. */
const char* dmuon_last_error(dmuon_handle_t h);

/* Bounded waits: how long a tensor-core kernel's pipeline wait may go without
 * progress before the kernel gives up, drains its own copies, frees its
 * tensor memory, returns, and dmuon_get_status reports DMUON_ERR_TIMEOUT.
 * ns == 0 restores the default (4 s).  Applies to later launches of the
 * handle; a tiny value makes the first non-immediate wait give up, which
 * is how the failure path is exercised without faulting the GPU. */
int dmuon_set_wait_timeout(dmuon_handle_t h, uint64_t ns);

/* Tensor-core tiling of later plans: 0 = automatic (the default: CTA pairs when
 * the device can co-schedule 2-CTA clusters, some chunked matrix has a short
 * side above 128 and the chunked matrices give at least one 256x256 Gram
 * super-tile per pair; single CTAs otherwise, with 128x128 tiles when the
 * 128x256 Gram tiles would number fewer than the SMs), 1 = single CTAs
 * computing 128x256 tiles, 2 = CTA pairs computing 256x256 tiles
 * (cta_group::2), 3 = single CTAs computing 128x128 tiles.  The result is the
 * same maths up to the order of the fp32 sums of a tile's products; the
 * choice only changes speed.  It applies to the direct backend; the Gram
 * backend always uses CTA pairs.  DMUON_ERR_UNSUPPORTED if pairs are
 * requested but unavailable, DMUON_ERR_ARG for another mode. */
int dmuon_set_tile_mode(dmuon_handle_t h, int mode);

/* Chunking of later plans: the matrix list is cut into contiguous chunks of
 * at most `elems` matrix elements (a larger matrix is a chunk of its own);
 * each chunk runs its whole launch sequence before the next starts, and all
 * chunks share one workspace sized for the largest.  0 selects the default
 * (2^29 elements); a value above the list's total gives one chunk.  The
 * result does not depend on the chunking. */
int dmuon_set_chunk_elements(dmuon_handle_t h, int64_t elems);

/* Overlap of later plans with two or more chunks (default off): chunk c+1's
 * momentum/normalisation pass runs on an internal stream while chunk c's
 * tensor-core phases run on the caller's stream; chunks then alternate
 * between two workspaces (twice the workspace memory).  The call stays
 * ordered on the caller's stream (fork and join through events).  The
 * result does not depend on the setting.  On a power-capped GB300 running
 * the Llama-3-8B set it measured the same step time either way. */
int dmuon_set_overlap(dmuon_handle_t h, int on);

/* How later plans deal each phase's work items (256 x 256 output tiles,
 * or 128-row halves) to the persistent CTAs or CTA pairs (default on):
 * on, longest first, each to the one with the least K-blocks so far, so a
 * list mixing long and short products (one Llama-3-8B layer: Grams with
 * K = 14336 and K = 4096) ends evenly; off, the sorted list round-robin.
 * The result is bitwise the same either way (each tile's arithmetic does not
 * depend on who computes it).  dmuon_plan_summary reports the balance. */
int dmuon_set_balanced_dealing(dmuon_handle_t h, int on);

/* Direct backend (chunked matrices), calls from now on: the number of
 * leading Newton-Schulz iterations whose products take fp16 operands (>= 1;
 * default 3; 64 or more: every iteration); later iterations take bf16 with
 * the same scales.  fp16 draws more power than bf16 at the same tensor-core
 * rate, so on a GB300 held at its power cap each bf16 iteration is slightly
 * faster; the first iterations carry most of the rounding error of inputs
 * with widely spread singular values.  DMUON_ERR_ARG for iters < 1. */
int dmuon_set_fp16_iterations(dmuon_handle_t h, int iters);

/* Direct backend, calls from now on: whether every Gram, Gram2 and Apply
 * product of every iteration of a chunk runs in ONE persistent launch instead
 * of one launch per phase and iteration.  mode 0: never; 1: always; 2
 * (default): for chunks whose three phases hold at most 8 work items per
 * persistent CTA (or CTA pair), where launch fills and drains dominate.  In
 * the fused launch each CTA (pair) runs, iteration by iteration and phase by
 * phase, the same dealt work items as the per-phase launches; before loading
 * a tile's operands it waits (bounded, like every wait of the kernels) until
 * its matrix's counter of finished tiles shows that matrix's previous phase
 * complete.  The result is bitwise the same either way.  Measured on GB300:
 * faster for small lists (TinyMLP d=512: 0.42 against 0.49 ms per step),
 * slower for large ones (Llama-3-8B set: 395 against 330 ms; its CTAs drift
 * apart across phases and read 41 % more from DRAM), hence the automatic
 * rule.  Needs every CTA of the launch resident at once (one per SM, as
 * launched): work on other streams only delays it, and a wait that runs out
 * reports DMUON_ERR_TIMEOUT.  DMUON_ERR_ARG for another mode. */
int dmuon_set_fused_phases(dmuon_handle_t h, int mode);

/* Small-matrix kernel for later plans (default on): every matrix whose
 * oriented shape has m = min(rows, cols) <= 128 and n = max(rows, cols) <= 512
 * (the TinyMLP projections of DMuon "Quick Start" at small widths; the
 * small parameters that "API Reference", section "Muon", packs together
 * under pack_small_params; 64x256 tensor-parallel shards) runs its whole step -- momentum, Nesterov input, norm, the ns_steps
 * iterations and the update -- in one CTA, with the iterate in shared memory
 * and the products in tensor memory; all such matrices share one launch.
 * Off: they run through the chunked tensor-core path like the others.  Same
 * maths and fp16 roundings either way (the summation order inside a product
 * differs, so results agree to rounding, not bitwise).  Returns
 * DMUON_ERR_UNSUPPORTED if it cannot be enabled on this device. */
int dmuon_set_small_path(dmuon_handle_t h, int on);

/* Kernel launches issued by this handle since creation (a counter). */
int64_t dmuon_launch_count(dmuon_handle_t h);

/*
 * Per-phase CUDA-event timing (the counterpart of the pages'
 * record_step_profile / consume_last_step_profile, DMuon "API Reference",
 * section "Muon").  While enabled, each launch is bracketed by events on
 * its stream.  dmuon_profile_read() synchronises, then adds the elapsed
 * milliseconds and launch counts per kernel kind into ms[k] and count[k]
 * for k < n_kinds (kinds: 0 momentum+norm, 1 norm finalise, 2 Gram X X^T,
 * 3 A*A, 4 B*X (+update), 5 update without NS, 6 AdamW, 7 clipping, the
 * last bracketing its whole launch sequence) and resets the record.
 */
#define DMUON_KIND_MOMENTUM 0
#define DMUON_KIND_FINALIZE 1
#define DMUON_KIND_GRAM     2
#define DMUON_KIND_GRAM2    3
#define DMUON_KIND_APPLY    4
#define DMUON_KIND_UPDATE0  5
#define DMUON_KIND_ADAMW    6
#define DMUON_KIND_CLIP     7
#define DMUON_KIND_SMALL    8
#define DMUON_KIND_GS_GRAM  9   /* Gram backend: R = kappa s^2 X X^T        */
#define DMUON_KIND_GS_PROD  10  /* Gram backend: m x m window products     */
#define DMUON_KIND_NS_FUSED 11  /* direct backend: every product of every
                                 * iteration of a chunk in one launch       */
#define DMUON_NUM_KINDS     12
int dmuon_profile_enable(dmuon_handle_t h, int on);
int dmuon_profile_read(dmuon_handle_t h, double* ms, int64_t* count,
                       int n_kinds);

/* Human-readable description of the current plan (matrices, work items
 * per phase, how evenly each phase's items are dealt to the persistent
 * CTAs or CTA pairs -- "balance": the busiest one's K-blocks over the mean,
 * 1 = even -- and workspace bytes) into buf (NUL-terminated, truncated to
 * len).  Returns the full length needed. */
int dmuon_plan_summary(dmuon_handle_t h, char* buf, size_t len);

/*
 * Polar Express coefficient table (DMuon "API Reference", section
 * "POLAR_EXPRESS_COEFFICIENTS": the Gram backend's default in the pages,
 * built by the method of arXiv:2505.16932 with a safety factor, values not
 * printed).  Row k is the odd quintic p(x) = a x + b x^3 + c x^5 with the
 * least max |1 - p(x)| over the interval of singular values that rows
 * 0..k-1 leave -- [lower, upper] for row 0, then [1 - E, 1 + E] with E the
 * previous row's least error -- then scaled by the safety factor s as
 * (a / s, b / s^3, c / s^5), i.e. p(x / s).  The pages' s is 1.05;
 * lower = 1e-3 and upper = 1 are this library's reading of the start.
 * Rows whose interval lies within 1e-7 of 1 (after about six steps from
 * [1e-3, 1]) take the construction's limit (15/8, -10/8, 3/8).
 *   out  host, 3 * steps floats, rows (a, b, c).
 * Host only (no device, no handle).  DMUON_ERR_ARG for steps outside
 * 1..DMUON_MAX_NS_STEPS, lower <= 0, upper <= lower, safety <= 0, a null
 * out, or an interval on which the exchange does not converge.
 */
int dmuon_polar_express_coefficients(int steps, double lower, double upper,
                                     double safety, float* out);

/*
 * The Gram-space backend's fp16 range check of a coefficient table (host
 * only): follows the largest singular value the iterate can reach (1 for
 * the normalised input, then max |p_k| over [0, u] after step k) and
 * bounds every fp16 buffer for all inputs -- the step factor Z, kappa R and
 * kappa R Z (kappa <= 1024) at half the fp16 maximum and each restart
 * window's factor (windows of at most two steps) at 8192.
 *   coeffs    host, 3 * ns_steps floats, or NULL for the backend's default
 *             (the Polar Express table of ns_steps rows).
 *   restarts  host, n_restarts entries, or NULL for {2}.
 *   why       host buffer of why_len bytes for the reason (may be NULL).
 * DMUON_OK if the table fits, DMUON_ERR_ARG otherwise (or for bad
 * arguments: ns_steps or n_restarts outside 0..DMUON_MAX_NS_STEPS, a null
 * restarts with n_restarts > 0, a non-finite coefficient).
 */
int dmuon_gram_check_coefficients(int ns_steps, const float* coeffs,
                                  const int* restarts, int n_restarts,
                                  char* why, size_t why_len);

/*
 * Host-only preview of the plan a handle would build for this list, without
 * a device: the tile kind the automatic choice (tile_mode 0) or the forced
 * one (1 single CTAs 128x256, 2 CTA pairs, 3 single CTAs 128x128) gives,
 * the chunks, the work items per
 * phase and how evenly they are dealt ("balance", as in
 * dmuon_plan_summary), for a device with `clusters` co-resident 2-CTA
 * clusters (0 = none) and `sms` SMs; balanced = 0 previews the strided
 * dealing.  The small-matrix kernel is assumed on.  Writes a NUL-terminated
 * summary into buf (truncated to len) and returns its full length, or
 * DMUON_ERR_ARG for bad arguments (the Gram backend needs clusters >= 1).
 */
int dmuon_plan_preview(const dmuon_shape_t* shapes, int n_mats, int backend,
                       int tile_mode, int clusters, int sms, int balanced,
                       char* buf, size_t len);

/* Static string for a status code. */
const char* dmuon_error_string(int code);

/* Library version string. */
const char* dmuon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DMUON_H */
