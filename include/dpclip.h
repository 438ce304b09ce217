/*
 * dpclip -- per-linear-layer DP-SGD clipping path for one GB300 (sm_103a).
 *
 * C ABI of libdpclip.so.  For one linear layer and a batch of B sequences of T
 * tokens, sample i has input activations A_i (T x d) and output gradients G_i
 * (T x p); its weight gradient is M_i = A_i^T G_i (d x p).  The library
 * computes
 *   - per-sample squared norms ||M_i||_F^2, exactly or with the randomized
 *     trace estimators Hutch and Hutch++,
 *   - clip scales s_i = min(1, C / n_i) with n_i the square root of a norm,
 *   - the clipped, noised sum  sum_i s_i M_i + N(0, sigma^2 C^2 I).
 *
 * Sources: "Technical summary: efficient DP-SGD for LLMs with randomized
 * clipping" (gist.science summary of arXiv 2605.24879), sections "Core
 * mechanism" and "Algorithmic flow"; the "DP-SGD" glossary entry of jisaku.com,
 * section "DP-SGD algorithm".
 *
 * Common conventions
 *   Layout   A is [B][T][d] and G is [B][T][p], row-major and contiguous.  The
 *            gradient output is [d][p] row-major fp32 (the transpose of a
 *            PyTorch nn.Linear weight gradient).
 *   dtype    DPCLIP_F32: A, G are float.  DPCLIP_BF16: A, G are bfloat16 and
 *            every product is accumulated in fp32; bf16 needs d % 8 == 0 and
 *            p % 8 == 0 (16-byte rows for the tensor-memory-access engine).
 *   Memory   every pointer argument is device memory owned by the caller and
 *            must stay valid until the stream reaches the work; A, G, grad and
 *            the workspace must be 16-byte aligned, the workspace 256-byte
 *            aligned.  The library never allocates, frees or synchronises
 *            (except dpclip_workspace_status, which synchronises by design).
 *            Scratch memory comes only from the caller's workspace, sized by
 *            dpclip_workspace_size; one workspace must not be used by two
 *            calls that can run at the same time.
 *   Streams  work is enqueued asynchronously on `stream` (NULL: legacy default
 *            stream) of the current CUDA device.
 *   Errors   arguments are checked on the host before anything is enqueued:
 *            a bad argument returns a negative status and enqueues nothing.
 *            Launch failures return DPCLIP_ERR_CUDA.  Device-side waits are
 *            bounded: a wait that expires makes the kernels stop early and
 *            records DPCLIP_ERR_TIMEOUT in the workspace, readable with
 *            dpclip_workspace_status.  No C++ exception crosses this ABI.
 *   Random   probes and noise come from Philox-4x32-10 (Salmon et al., SC'11)
 *            keyed by `seed`; element e of stream s uses counter
 *            (e / 4, s, offset_lo, offset_hi) and lane e % 4 through a
 *            Box-Muller transform.  Streams: 0 = Hutch probe P, 1 = Hutch++
 *            sketch S, 2 = Hutch++ tail probes G', 3 = gradient noise.  The
 *            same (seed, offset) always gives the same numbers; pass the step
 *            index as `offset`.
 */
#ifndef DPCLIP_H
#define DPCLIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dpclip_stream_t;   /* same type as cudaStream_t */

enum dpclip_status {
  DPCLIP_OK = 0,
  DPCLIP_ERR_INVALID_ARG = -1,   /* null pointer, non-positive size, bad enum */
  DPCLIP_ERR_UNSUPPORTED = -2,   /* valid but not supported: alignment, k range */
  DPCLIP_ERR_WORKSPACE = -3,     /* workspace missing, misaligned or too small */
  DPCLIP_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
  DPCLIP_ERR_TIMEOUT = -5        /* a device-side wait expired (see status) */
};

enum dpclip_dtype { DPCLIP_F32 = 0, DPCLIP_BF16 = 1 };

enum dpclip_exact_method {
  DPCLIP_EXACT_AUTO = 0,    /* direct when 2*d*p < T*(d+p) (fewer flops), else ghost */
  DPCLIP_EXACT_GHOST = 1,   /* sum((A_i A_i^T) o (G_i G_i^T)) */
  DPCLIP_EXACT_DIRECT = 2   /* ||A_i^T G_i||_F^2, tile by tile, never stored */
};

/* Probe law of the randomized estimators.  Gaussian: i.i.d. N(0,1) ("Core
 * mechanism", item 1).  Rademacher: i.i.d. {+1, -1}, the alternative sketch
 * the summary names as future work; exact in bfloat16.  Element e of a
 * Rademacher stream is -1 when the top bit of word e % 4 of its Philox block
 * (the same counter as for the normals) is set, +1 otherwise. */
enum dpclip_probe { DPCLIP_PROBE_GAUSSIAN = 0, DPCLIP_PROBE_RADEMACHER = 1 };

enum dpclip_op {
  DPCLIP_OP_NORMS_EXACT = 0,
  DPCLIP_OP_NORMS_HUTCH = 1,
  DPCLIP_OP_NORMS_HUTCHPP = 2,
  DPCLIP_OP_CLIPPED_NOISY_GRAD = 3,
  DPCLIP_OP_STORED_DIRECT = 4,   /* dpclip_norms_direct_store + dpclip_stored_clipped_noisy_grad */
  DPCLIP_OP_BIAS = 5             /* dpclip_bias_grads (d and param ignored) */
};

/* Largest probe count k for Hutch (k <= 32) and Hutch++ (k - floor(k/3) <= 32). */
#define DPCLIP_HUTCH_MAX_K 32
#define DPCLIP_HUTCHPP_MAX_K 48

/* Workspace bytes for one call of `op` on these sizes.  `param` is k for the
 * Hutch/Hutch++ ops, the dpclip_exact_method for DPCLIP_OP_NORMS_EXACT and
 * ignored for the gradient.  Writes *bytes; returns a status. */
int dpclip_workspace_size(int op, int B, int T, int d, int p, int dtype, int param,
                          size_t* bytes);

/* Exact per-sample squared norms sqnorms[i] = ||A_i^T G_i||_F^2 (fp32 [B]).
 * Ghost form: "Problem definition" (ghost clipping, T^2 memory) and the trace
 * identity of "Core mechanism"; direct form: the per-sample gradient itself,
 * reduced tile by tile. */
int dpclip_norms_exact(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                       int method, float* sqnorms, void* ws, size_t ws_bytes,
                       dpclip_stream_t stream);

/* Hutch estimate ("Core mechanism", item 1): with P (p x k) i.i.d. N(0,1),
 * one P per call shared by all samples, sqnorms[i] = (1/k) ||A_i^T (G_i P)||_F^2.
 * bf16: P is rounded to bfloat16.  1 <= k <= DPCLIP_HUTCH_MAX_K. */
int dpclip_norms_hutch(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                       int k, uint64_t seed, uint64_t offset, float* sqnorms, void* ws,
                       size_t ws_bytes, dpclip_stream_t stream);

/* Hutch++ estimate ("Core mechanism", item 2) with a budget of k products:
 * r = floor(k/3) sketch columns S, Q = orthonormal basis of O_i S (computed
 * per sample), head = trace(Q^T O_i Q), W = (I - Q Q^T) G' with m = k - 2r
 * tail probes, sqnorms[i] = head + trace(W^T O_i W) / m, where
 * O_i = G_i^T A_i A_i^T G_i.  3 <= k <= DPCLIP_HUTCHPP_MAX_K. */
int dpclip_norms_hutchpp(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                         int k, uint64_t seed, uint64_t offset, float* sqnorms, void* ws,
                         size_t ws_bytes, dpclip_stream_t stream);

/* dpclip_norms_hutch / dpclip_norms_hutchpp with a choice of probe law
 * (dpclip_probe); the plain entry points use DPCLIP_PROBE_GAUSSIAN.  Same
 * workspace sizes.  An unknown probe value returns DPCLIP_ERR_INVALID_ARG. */
int dpclip_norms_hutch_ex(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                          int k, int probe, uint64_t seed, uint64_t offset, float* sqnorms,
                          void* ws, size_t ws_bytes, dpclip_stream_t stream);
int dpclip_norms_hutchpp_ex(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                            int k, int probe, uint64_t seed, uint64_t offset, float* sqnorms,
                            void* ws, size_t ws_bytes, dpclip_stream_t stream);

/* Clipped noisy gradient ("DP-SGD algorithm" steps 3-4; "Algorithmic flow"
 * steps 4-5):
 *   s_i  = min(1, C / sqrt(sqnorms[i])), s_i = 1 when sqnorms[i] == 0,
 *   grad = sum_i s_i A_i^T G_i + sigma * C * Z,   Z ~ N(0, I) from stream 3,
 *          entry (r, c) of grad using element index r * p + c.
 * sqnorms (fp32 [B], device) may be the sum over several layers.  grad is fp32
 * [d][p].  scales (fp32 [B]) and clipped (uint8 [B], 1 when sqrt(sqnorms[i]) >
 * C) are optional outputs (NULL to skip).  C > 0, sigma >= 0.  The 1/|B| of
 * the SGD update is not applied. */
int dpclip_clipped_noisy_grad(const void* A, const void* G, int B, int T, int d, int p,
                              int dtype, const float* sqnorms, float C, float sigma,
                              uint64_t seed, uint64_t offset, float* grad, float* scales,
                              uint8_t* clipped, void* ws, size_t ws_bytes,
                              dpclip_stream_t stream);

/* Exact per-sample squared norms by the direct method, keeping every
 * per-sample gradient M_i = A_i^T G_i (fp32) in `ws` for
 * dpclip_stored_clipped_noisy_grad.  This is the per-sample gradient
 * materialisation of "Problem definition" taken as a deliberate trade: it
 * costs B*d*p*4 bytes of workspace (268 MB for B = 4 at d x p = 2048 x 8192,
 * small against this GPU's HBM), and in return the clipped sum is one
 * elementwise pass over the stored gradients instead of a second GEMM over A
 * and G.  accumulate = 0: sqnorms[i] = ||M_i||_F^2; accumulate = 1:
 * sqnorms[i] += ||M_i||_F^2 (the per-sample norm of a whole model is the sum
 * over its layers).  Workspace: dpclip_workspace_size(DPCLIP_OP_STORED_DIRECT,
 * ...), param ignored; its contents must be kept, unchanged, until the
 * matching dpclip_stored_clipped_noisy_grad has been enqueued. */
int dpclip_norms_direct_store(const void* A, const void* G, int B, int T, int d, int p,
                              int dtype, int accumulate, float* sqnorms, void* ws,
                              size_t ws_bytes, dpclip_stream_t stream);

/* The clipped noisy gradient of dpclip_clipped_noisy_grad (same formula, the
 * same noise stream and element mapping, the same optional outputs) from the
 * per-sample gradients a dpclip_norms_direct_store call with the same B, d
 * and p left in `ws`, enqueued after it on the same stream.  sqnorms may
 * hold the sum over several layers.  grad: 16-byte aligned. */
int dpclip_stored_clipped_noisy_grad(int B, int d, int p, const float* sqnorms, float C,
                                     float sigma, uint64_t seed, uint64_t offset, float* grad,
                                     float* scales, uint8_t* clipped, const void* ws,
                                     size_t ws_bytes, dpclip_stream_t stream);

/* Per-sample gradients of the bias of a linear layer y_t = x_t W + b: the
 * derivative of y_t with respect to b is the identity, so
 * bias_grads[i][c] = sum_t G_i[t][c] (fp32 [B][p], device, may be NULL), and
 * the bias's share of the per-sample squared norm ("DP-SGD algorithm" step 3
 * clips the gradient of every parameter): sqnorms[i] = ||b_i||^2
 * (accumulate = 0) or sqnorms[i] += ||b_i||^2 (accumulate = 1; sqnorms may be
 * NULL).  G as for the norms ([B][T][p], bf16 or fp32).  Reads G once.
 * Workspace: dpclip_workspace_size(DPCLIP_OP_BIAS, B, T, 0, p, dtype, 0). */
int dpclip_bias_grads(const void* G, int B, int T, int p, int dtype, int accumulate,
                      float* sqnorms, float* bias_grads, void* ws, size_t ws_bytes,
                      dpclip_stream_t stream);

/* Clipped noisy bias gradient: s_i = min(1, C / sqrt(sqnorms[i])) (1 when 0),
 * grad_b[c] = sum_i s_i bias_grads[i][c] + sigma * C * z_c with z from Philox
 * stream 4 at element c (its own stream: the weight noise is stream 3).
 * sqnorms should be the whole per-sample squared norm (weights and bias).
 * bias_grads as written by dpclip_bias_grads; grad_b fp32 [p].  B <= 12288. */
int dpclip_clipped_noisy_bias_grad(const float* bias_grads, int B, int p, const float* sqnorms,
                                   float C, float sigma, uint64_t seed, uint64_t offset,
                                   float* grad_b, dpclip_stream_t stream);

/* Parameter update fused into the gradient calls ("DP-SGD algorithm" step 5:
 * theta <- theta - eta * g / L, g the noisy clipped sum).  `param` is the
 * layer's fp32 parameter tensor in the gradient's layout ([d][p] weights or
 * [p] bias, device, 16-byte aligned for the weights); it is updated in place
 * as param -= (lr / denom) * g.  denom is the lot size L of the average: the
 * drawn lot size, or its expectation when the lot is Poisson sampled (then
 * the drawn B varies per step, may be 0, and the update's noise scale stays
 * sigma C lr / L).  store_grad = 0 skips writing g itself (grad may then be
 * NULL on the bf16 paths). */
typedef struct dpclip_sgd_update {
  float* param;
  float lr;
  float denom;
  int store_grad;
} dpclip_sgd_update;

/* dpclip_clipped_noisy_grad, dpclip_stored_clipped_noisy_grad and
 * dpclip_clipped_noisy_bias_grad with an optional fused update (NULL: none)
 * and with B = 0 accepted (an empty lot: A, G, sqnorms and the stored
 * gradients are not read, g = sigma C z).  fp32 inputs need `grad` even with
 * store_grad = 0 (it is the scratch of the update). */
int dpclip_clipped_noisy_grad_ex(const void* A, const void* G, int B, int T, int d, int p,
                                 int dtype, const float* sqnorms, float C, float sigma,
                                 uint64_t seed, uint64_t offset, float* grad, float* scales,
                                 uint8_t* clipped, const dpclip_sgd_update* update, void* ws,
                                 size_t ws_bytes, dpclip_stream_t stream);
int dpclip_stored_clipped_noisy_grad_ex(int B, int d, int p, const float* sqnorms, float C,
                                        float sigma, uint64_t seed, uint64_t offset, float* grad,
                                        float* scales, uint8_t* clipped,
                                        const dpclip_sgd_update* update, const void* ws,
                                        size_t ws_bytes, dpclip_stream_t stream);
int dpclip_clipped_noisy_bias_grad_ex(const float* bias_grads, int B, int p, const float* sqnorms,
                                      float C, float sigma, uint64_t seed, uint64_t offset,
                                      float* grad_b, const dpclip_sgd_update* update,
                                      dpclip_stream_t stream);

/* FIBER ("Technical summary: FIBER", Method A and C): the privatized gradient
 * g = grad / denom is filtered in innovation space, nu = g - gf,
 * r = (1 - omega) r + omega nu, gf = gf + r, and AdamW runs on gf with the
 * bias-corrected second moment reduced by the filtered noise variance,
 * vbar = max(vhat - A(omega) noise_var, eps_v), A(omega) = (2 - omega) /
 * (4 - 3 omega):  param -= lr (mhat / (sqrt(vbar) + eps) + weight_decay param).
 * All tensors fp32 in the gradient's layout, device, updated in place; the
 * four states start at zero before step 1.  0 < omega <= 1, step >= 1,
 * denom > 0, noise_var >= 0 (for the clipped noisy sum of this library,
 * (sigma C / denom)^2).  param/filt/resid/m/v 16-byte aligned for the weights. */
typedef struct dpclip_fiber_adamw {
  float* param;
  float* filt;
  float* resid;
  float* m;
  float* v;
  float lr, beta1, beta2, eps, eps_v, weight_decay;
  float omega;
  float noise_var;
  float denom;
  int step;
} dpclip_fiber_adamw;

/* One FIBER step on n parameters from a gradient already formed (grad fp32
 * [n], device). */
int dpclip_fiber_adamw_step(const float* grad, int64_t n, const dpclip_fiber_adamw* opt,
                            dpclip_stream_t stream);

/* The gradient calls followed by the FIBER step.  The stored-tile and bias
 * calls fuse it into the pass that forms the gradient (grad / grad_b may
 * then be NULL: not stored).  The GEMM call writes `grad` (required) and runs
 * the step as one more pass over it: inside the GEMM epilogue the five state
 * streams per element cost more than a separate HBM-bound pass.  B = 0 as
 * for the _ex calls. */
int dpclip_clipped_noisy_grad_fiber(const void* A, const void* G, int B, int T, int d, int p,
                                    int dtype, const float* sqnorms, float C, float sigma,
                                    uint64_t seed, uint64_t offset, float* grad, float* scales,
                                    uint8_t* clipped, const dpclip_fiber_adamw* opt, void* ws,
                                    size_t ws_bytes, dpclip_stream_t stream);
int dpclip_stored_clipped_noisy_grad_fiber(int B, int d, int p, const float* sqnorms, float C,
                                           float sigma, uint64_t seed, uint64_t offset,
                                           float* grad, float* scales, uint8_t* clipped,
                                           const dpclip_fiber_adamw* opt, const void* ws,
                                           size_t ws_bytes, dpclip_stream_t stream);
int dpclip_clipped_noisy_bias_grad_fiber(const float* bias_grads, int B, int p,
                                         const float* sqnorms, float C, float sigma,
                                         uint64_t seed, uint64_t offset, float* grad_b,
                                         const dpclip_fiber_adamw* opt, dpclip_stream_t stream);

/* Clip scales alone: scales[i] = min(1, C / sqrt(sqnorms[i])) (1 when the norm
 * is 0) and clipped[i] = sqrt(sqnorms[i]) > C; either output may be NULL. */
int dpclip_clip_scales(const float* sqnorms, int B, float C, float* scales, uint8_t* clipped,
                       dpclip_stream_t stream);

/* The n standard normals of one Philox stream (see "Random" above), written
 * as float (dtype DPCLIP_F32) or rounded to bfloat16 (DPCLIP_BF16) into `out`
 * (device, 4-byte aligned). */
int dpclip_philox_normal(void* out, int64_t n, int dtype, uint64_t seed, uint32_t stream_id,
                         uint64_t offset, dpclip_stream_t stream);

/* Size of the library-owned scratch array behind dpclip_norms_hutch_noalloc
 * (16 MiB; covers Hutch with k <= 32 at B*T = 16384 tokens and d, p up to
 * 2048 x 8192, for example). */
#define DPCLIP_NOALLOC_SCRATCH_BYTES (16u << 20)

/* dpclip_norms_hutch without a caller workspace and without any allocation.
 * The pages have no counterpart for this: it exists for callers that cannot
 * allocate device memory where they need the norms (a host framework calling
 * from a callback in which device allocation is forbidden after set-up, a
 * process whose device memory is all handed out by another allocator, a
 * latency-critical loop where an allocation could stall on the device).
 * Arguments and result as dpclip_norms_hutch.  Scratch is a library-owned
 * device array of DPCLIP_NOALLOC_SCRATCH_BYTES, created on every GPU that
 * loads the library and held until the process exits.  Sizes whose Hutch
 * workspace (dpclip_workspace_size) exceeds it return DPCLIP_ERR_WORKSPACE
 * before anything is enqueued.  The first call on a device looks up the
 * array's device address with that device current; make that first call
 * before any stream capture.  The address is kept per device and context: a
 * device reset (cudaDeviceReset) destroys the array, and the first call in
 * the new context looks the address up again.  Every call shares the array
 * and it keeps the last call's contents (each call clears what must start at
 * zero): calls that can overlap on the GPU race on it, so issue them on one
 * stream.  Never calls cudaMalloc, cudaFree or any allocating routine.  A
 * bounded wait that expires on the device is not reported by the return
 * value (the call returns once its kernels are enqueued): read it with
 * dpclip_noalloc_status. */
int dpclip_norms_hutch_noalloc(const void* A, const void* G, int B, int T, int d, int p,
                               int dtype, int k, uint64_t seed, uint64_t offset, float* sqnorms,
                               dpclip_stream_t stream);

/* Synchronises `stream`, then returns DPCLIP_OK or the error that the device
 * recorded in the scratch array of dpclip_norms_hutch_noalloc on the current
 * device (DPCLIP_ERR_TIMEOUT: a bounded wait expired and the norms of that
 * call are not valid), or DPCLIP_ERR_CUDA if the synchronisation or the read
 * failed.  The array is shared, so this is the status of the last call that
 * ran on it.  Allocates nothing. */
int dpclip_noalloc_status(dpclip_stream_t stream);

/* The n Rademacher values of one Philox stream (see dpclip_probe), written as
 * float or bfloat16 into `out` (device, 4-byte aligned). */
int dpclip_philox_rademacher(void* out, int64_t n, int dtype, uint64_t seed, uint32_t stream_id,
                             uint64_t offset, dpclip_stream_t stream);

/* Synchronises `stream`, then returns DPCLIP_OK or the error the device
 * recorded in the workspace of the last call that used it
 * (DPCLIP_ERR_TIMEOUT), or DPCLIP_ERR_CUDA if the synchronisation failed. */
int dpclip_workspace_status(const void* ws, dpclip_stream_t stream);

/* Test hook for the bounded-wait path: enqueues one kernel whose barrier wait
 * is never satisfied, with a limit of `timeout_us` microseconds (1..10^6); the
 * kernel gives up, records DPCLIP_ERR_TIMEOUT in `ws` and returns.  Follow
 * with dpclip_workspace_status. */
int dpclip_selftest_wait_timeout(void* ws, size_t ws_bytes, int timeout_us,
                                 dpclip_stream_t stream);

/* Host-only diagnostic (no device work): the schedule that
 * dpclip_clipped_noisy_grad gives the tiles left after the full waves, for
 * `pairs` CTA pairs, `ntiles` pair tiles of 256 x 256, B samples of `tblocks`
 * 64-token blocks.  Writes *waves (full waves of whole tiles) and *ntail
 * (tiles left).  Each segment is 5 int64 at segs[5 j]: pair, tail tile,
 * first and end K-block of the tile's time line (sample i's block kb is
 * i * tblocks + kb) and the workspace slot; pairs appear in index order and
 * a pair's segments in the order it runs them.  Each contribution is 2 int64
 * at contrib[2 j]: tail tile and slot, per tile in the order the partial
 * sums are added.  *nsegs and *ncontrib receive the full counts; records
 * beyond seg_cap or contrib_cap are not written.  DPCLIP_ERR_INVALID_ARG for
 * pairs outside 1..80 or non-positive sizes. */
int dpclip_grad_tail_schedule(int pairs, int ntiles, int B, int tblocks, int* waves, int* ntail,
                              int64_t* segs, int seg_cap, int* nsegs, int64_t* contrib,
                              int contrib_cap, int* ncontrib);

/* Host-only diagnostic (no device work): how dpclip_norms_exact's ghost form
 * deals its work units (sample, 256-token tile pair a' <= b') over `pairs`
 * CTA pairs (grids of fewer pairs than units; the call uses min(resident
 * pairs, units)).  *nfull units are dealt whole, round-robin; each of the
 * B * units - *nfull others is cut along p into *tail_split slices of
 * *pb_per_split 64-column blocks (the last one shorter), and, when
 * *tail_shared is 1, one more sub-unit that forms the unit's A Gram block
 * once for the slices (else every slice recomputes it).
 * DPCLIP_ERR_INVALID_ARG for pairs outside 1..80, non-positive sizes or
 * null outputs. */
int dpclip_ghost_schedule(int pairs, int B, int T, int d, int p, int* nfull, int* tail_split,
                          int* pb_per_split, int* tail_shared);

/* Human-readable name of a status code. */
const char* dpclip_status_string(int status);

/* Library version string. */
const char* dpclip_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DPCLIP_H */
