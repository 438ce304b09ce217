// Internal interface between the C-ABI layer (dpclip.cu) and the kernel
// translation units.  Host-side only types plus CUtensorMap.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "../../include/dpclip.h"

namespace dpclip {

// Launches `kernel` with programmatic stream serialisation, so that its
// prologue overlaps the tail of the previous kernel in the stream (the kernel
// itself waits for that kernel before touching global memory).  A cluster
// with cluster.x > 0 groups CTAs into thread-block clusters of those
// dimensions; cluster.x == 0 launches without a cluster attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, dim3 cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster.x;
  attr[1].val.clusterDim.y = cluster.y;
  attr[1].val.clusterDim.z = cluster.z;
  cfg.attrs = attr;
  cfg.numAttrs = cluster.x > 0 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with clusters of cluster_x consecutive CTAs along x (none when
// cluster_x <= 0).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int cluster_x, Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, s,
                            cluster_x > 0 ? dim3((unsigned)cluster_x, 1, 1) : dim3(0, 0, 0),
                            std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------
// Tile geometry of the tensor-core kernels
// ----------------------------------------------------------------------------
constexpr int kTokTileM = 128;     // tokens per tok_gemm tile
constexpr int kFeatTileM = 128;    // features per feat_gemm tile
constexpr int kBlockK = 64;        // bf16 elements per 128-byte swizzled row
constexpr int kDpTileM = 128;      // d rows per CTA of a gradient / direct-norm pair tile (256)
constexpr int kDpTileN = 256;      // p columns per gradient / direct-norm tile
constexpr int kGhostTile = 128;    // tokens per CTA of a ghost Gram pair tile (256 x 256)
constexpr int kEpiWarps = 8;       // epilogue warps of the persistent kernels
constexpr int kMaxNP = 32;         // widest skinny operand (probe columns)
constexpr int kMaxSplits = 8;      // K-splits of a skinny tile (one portable cluster)

// Skinny-GEMM epilogue modes of feat_gemm.
enum FeatMode { kFeatOutF32 = 0, kFeatOutHiLo = 1, kFeatSqNorm = 2 };

// tok_gemm:  out[i][j][t] = sum_f X[i][t][f] * W[w(i)][j][f]
//   X: [B][T][F] bf16 (K-major operand), W: [Bw][NP][F] bf16 hi (+ lo).
//   Output: hi/lo bf16 [B][NP][Tp], Tp = mtiles * 128 (rows >= T are zero).
struct TokGemmParams {
  CUtensorMap map_x;     // box {64, 128, 1}
  CUtensorMap map_whi;   // box {64, NP, 1}
  CUtensorMap map_wlo;   // box {64, NP, 1}
  int B, T, F, NP;
  int w_per_sample, has_lo;
  int mtiles, kblocks, splits, kb_per_split, Tp;
  int x_stream;          // X is read once: its loads evict first from L2
  __nv_bfloat16* out_hi;
  __nv_bfloat16* out_lo;
  uint32_t* err;
};

// feat_gemm: Z[i][f][j] = sum_t X[i][t][f] * Y[i][j][t]
//   X: [B][T][F] bf16 (MN-major operand), Y: [B][NP][Tp] bf16 hi + lo.
//   Modes: fp32 out [B][NP][F]; hi/lo bf16 out [B][NP][F];
//          sqnorm: sq[i] = sum_{f,j} w[j] * Z[i][f][j]^2.
struct FeatGemmParams {
  CUtensorMap map_x;     // box {64, 64, 1}
  CUtensorMap map_yhi;   // box {64, NP, 1}
  CUtensorMap map_ylo;
  int B, T, F, NP, Tp;
  int ftiles, tblocks, splits, tb_per_split, Fp;
  float w[kMaxNP];       // column weights for the sqnorm mode
  float* out_f32;
  __nv_bfloat16* out_hi;
  __nv_bfloat16* out_lo;
  float* sq;             // [B] output of the sqnorm mode
  float* qpart;          // [B][ftiles][splits]: each CTA's share of the square sum
  uint32_t* counters;    // [B]: CTAs of the sample done (sqnorm mode)
  int x_stream;          // X is read once: its loads evict first from L2 ...
  int x_keep_t0;         // ... except tokens >= x_keep_t0, which the next sweep reads first
  uint32_t* err;
};

// gemm_dp: per output tile (128 d x 256 p) and sample i, acc_i = A_i^T G_i.
//   grad mode:  grad = sum_i s_i acc_i + sigma*C*Z  (stored fp32 [d][p])
//   norm mode:  part[(tile*B + i)*8 + w] = partial sum of acc_i^2
// FIBER step on device (see dpclip_fiber_adamw): per element,
// g = grad * inv_denom, then the innovation filter and calibrated AdamW.
struct FiberDev {
  float* param;
  float* filt;
  float* resid;
  float* m;
  float* v;
  float lr, beta1, beta2, eps, eps_v, wd, omega;
  float calib;        // A(omega) * noise_var
  float inv_denom;
  float bc1, bc2;     // 1 / (1 - beta^t)
};

struct GemmDpParams {
  CUtensorMap map_a;     // A [B][T][d], box {64, 64, 1}
  CUtensorMap map_g;     // G [B][T][p], box {64, 64, 1}
  int B, T, d, p;
  int mtiles, ntiles, tblocks;   // mtiles: 128-row CTA tiles along d (even: pairs of them)
  // grad-mode schedule (set by launch_gemm_dp)
  int waves, ntail;      // full waves of whole pair tiles; pair tiles left after them
  uint32_t tail_cover;   // band levels of the tail schedule that cover (bit per level)
  float* slots;          // partial CTA tiles of 128 x 256 fp32, 2 per tail contribution
  uint32_t* tickets;     // [mtiles * ntiles] (CTA tiles), zero at launch
  const float* sqnorms;
  float C, sigma;
  uint64_t seed, offset;
  float* grad;
  float* scales;
  uint8_t* clipped;
  float* part;
  float* sq;             // norm mode: per-sample result [B]
  uint32_t* ticket;      // norm mode: zeroed grid ticket
  uint32_t* err;
  float* pstore;         // norm mode: if set, every tile A_i^T G_i also goes to [B][d][p]
  int accumulate;        // norm mode: sq[i] += the estimate (else =)
  float* upd_param;      // grad mode: if set, upd_param -= upd_scale * grad (grad may be null)
  float upd_scale;
};

// ghost: per sample i and 256-token tiles a' <= b', sum((A_a' A_b'^T) o
//   (G_a' G_b'^T)) over 128 x 128 blocks weighted 2 above the diagonal, 1 on
//   it; part[(g*2 + rank)*8 + w] per work item g, CTA rank and epilogue warp.
struct GhostParams {
  CUtensorMap map_a;     // box {64, 128, 1}
  CUtensorMap map_g;     // box {64, 128, 1}
  int B, T, d, p;
  int npairs, dblocks, pblocks;   // npairs: units (a', b') per sample
  int nfull;             // units dealt whole (a multiple of the grid of pairs)
  int tail_split, pb_per_split;   // the remaining units cut along p
  // tail_shared = 1: each remaining unit is one X sub-unit (X over d, stored
  // to xbuf) and tail_split Y sub-units that read it back; else every
  // sub-unit recomputes X
  int tail_shared;
  float* xbuf;           // [remaining units][2][128][256] fp32 (tail_shared)
  uint32_t* xready;      // [remaining units][2][8], zero at launch (tail_shared)
  float* part;           // [nfull + (B*npairs - nfull) * (tail_split + tail_shared)][2][8]
  float* sq;             // per-sample result [B]
  uint32_t* ticket;      // zeroed grid ticket
  uint32_t* err;
};

// Hutch++ middle step: per sample, orthonormal basis Q of V (p x r) by
// CholeskyQR2 (fp32, dependent columns dropped), W = G' - Q (Q^T G'), output [Q | W] padded to
// 32 columns, as hi/lo bf16 or fp32, [B][32][p].  Cooperative launch.
struct HppQrParams {
  const float* V;        // [B][ldv][p] fp32, columns j < r used
  int ldv;
  const void* Gp;        // [m][p], bf16 or fp32 (gp_bf16)
  int gp_bf16;
  int B, p, r, m;
  int cs;                // set by the launcher: CTAs (one cluster) per sample
  __nv_bfloat16* out_hi; // bf16 output (when out_f32 == nullptr)
  __nv_bfloat16* out_lo;
  float* out_f32;        // fp32 output [B][32][p]
  uint32_t* err;
  int gram_f64;          // first pass's Gram, Cholesky and inverse in fp64 (fp32 inputs)
};

// Generic fp32 SIMT GEMM over a batch:  acc[b](m,n) = sum_k X[b](m,k) Y[b](k,n)
// with arbitrary element strides; epilogue modes below.
enum SimtMode { kSimtStore = 0, kSimtSqNorm = 1, kSimtDotWith = 2, kSimtGrad = 3 };
struct SimtParams {
  const float* X;
  const float* Y;
  long long xb, xm, xk;
  long long yb, yk, yn;
  int batch, M, N, K;
  // store / dot-with operand
  float* out;
  long long ob, om, on;
  // sqnorm / dot-with partials: part[b * nblocks + block]
  float* part;
  float w[64];            // column weights (sqnorm)
  // grad
  const float* sqnorms;
  float C, sigma;
  uint64_t seed, offset;
  float* scales;
  uint8_t* clipped;
};

// ----------------------------------------------------------------------------
// Launchers (defined in the kernel translation units).  Each returns a
// cudaError_t from the launch.
// ----------------------------------------------------------------------------
cudaError_t launch_tok_gemm(const TokGemmParams& p, cudaStream_t s);
cudaError_t launch_feat_gemm(const FeatGemmParams& p, int mode, cudaStream_t s);
// Sizes the grid (CTA pairs) and, in grad mode, the schedule fields of p.
cudaError_t launch_gemm_dp(const GemmDpParams& p, bool grad_mode, cudaStream_t s);
// Sizes the grid (CTA pairs) and the tail schedule of p.
cudaError_t launch_ghost(const GhostParams& p, cudaStream_t s);
// Clusters of two CTAs of `kernel` that fit on the device at once (cached per
// device and slot: 0 gradient, 1 direct norms, 2 stored norms, 3 ghost).
constexpr int kPairSlots = 4;
int max_resident_pairs(const void* kernel, int threads, size_t smem, int slot);
cudaError_t launch_hpp_qr(const HppQrParams& p, cudaStream_t s);
cudaError_t launch_simt(const SimtParams& p, int mode, cudaStream_t s, int* nblocks_out);
int simt_nblocks(int M, int N);

// kind: DPCLIP_PROBE_GAUSSIAN or DPCLIP_PROBE_RADEMACHER.  Also clears
// `zero_words` 32-bit words at `zero` (the control block of a multi-kernel
// call) when zero != nullptr.
cudaError_t launch_philox_fill(void* out, int64_t rows, int64_t cols, int64_t rows_valid,
                               bool bf16, uint64_t seed, uint32_t stream_id, uint64_t offset,
                               cudaStream_t s, uint32_t* zero = nullptr, int zero_words = 0,
                               int kind = 0);
// Two fills (same columns, seed, offset and kind) in one launch.
cudaError_t launch_philox_fill2(void* out0, int64_t rows0, int64_t valid0, uint32_t stream0,
                                void* out1, int64_t rows1, int64_t valid1, uint32_t stream1,
                                int64_t cols, bool bf16, uint64_t seed, uint64_t offset,
                                cudaStream_t s, uint32_t* zero, int zero_words, int kind);
// Zeroes n control words after the stream's previous kernel (programmatic launch).
cudaError_t launch_clear_words(uint32_t* w, int n, cudaStream_t s);
cudaError_t launch_clip_scales(const float* sq, int B, float C, float* scales, uint8_t* clipped,
                               cudaStream_t s);
// sq[i] = scale * sum_{u < nunits, w < nw} part[(u * su + i * si) * nw + w]
// grad[e] = sum_i s_i M_i[e] + nscale z_e (z: Philox stream 3, element e), e < n,
// M_i = M + i * stride (stride a multiple of 4, M and grad 16-byte aligned),
// s_i = min(1, C / sqrt(sq[i])) (1 for sq[i] = 0); scales and clipped (either
// may be null) get s_i and [sqrt(sq[i]) > C].  B <= kMaxStoredB.
constexpr int kMaxStoredB = 12288;
cudaError_t launch_stored_grad(const float* M, int B, long long n, long long stride,
                               const float* sq, float C, float nscale, uint64_t seed,
                               uint64_t offset, float* grad, float* scales, uint8_t* clipped,
                               float* param, float upd_scale, const FiberDev* fiber,
                               cudaStream_t s);
// FIBER step over n elements of grad (fp32).
cudaError_t launch_fiber(const float* grad, long long n, const FiberDev& f, cudaStream_t s);
// grad (may be null) = nscale z (stream_id, element e), param (may be null)
// -= upd_scale * that, e < n: the gradient of an empty lot.
cudaError_t launch_noise_only(float* grad, float* param, long long n, float nscale,
                              float upd_scale, uint64_t seed, uint32_t stream_id, uint64_t offset,
                              const FiberDev* fiber, cudaStream_t s);
// param[e] -= scale * grad[e], e < n.
cudaError_t launch_sgd_update(float* param, const float* grad, long long n, float scale,
                              cudaStream_t s);
// Bias of the linear layer: bias[i][c] = sum_t G_i[t][c] (bias may be null),
// sq[i] (+)= ||bias_i||^2 (sq may be null); part holds bias_part_floats
// floats.  bias_clip: grad_b = sum_i s_i bias_i + nscale z (Philox stream 4).
size_t bias_part_floats(int B, int T, int p);
cudaError_t launch_bias_grads(const void* G, bool bf16, int B, int T, int p, float* part,
                              float* bias, float* sq, int accumulate, cudaStream_t s);
cudaError_t launch_bias_clip(const float* bias, int B, int p, const float* sq, float C, float nscale,
                             uint64_t seed, uint64_t offset, float* grad_b, float* param,
                             float upd_scale, const FiberDev* fiber, cudaStream_t s);
// part[i * nblk + b] = sum of squares of chunk b of M_i (n elements at M + i * stride).
cudaError_t launch_stored_sqnorm(const float* M, int B, long long n, long long stride, int nblk,
                                 float* part, cudaStream_t s);
cudaError_t launch_finalize_norms(const float* part, int B, int nunits, long long su,
                                  long long si, int nw, float scale, float* sq, cudaStream_t s,
                                  int accumulate = 0);
cudaError_t launch_noise_add(float* grad, long long n, float scale, uint64_t seed,
                             uint64_t offset, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s);

// Shared-memory footprint of each tensor-core kernel (bytes of dynamic smem).
size_t tok_gemm_smem(int NP);
size_t feat_gemm_smem(int NP);
size_t gemm_dp_smem();
size_t gemm_dp_slot_bytes(int max_grid);
void plan_grad_schedule(int ntiles, int B, int tblocks, int grid, int& waves, int& ntail,
                        uint32_t& cover);
// Summary of a tail schedule (host walk of grad_tail.cuh).
struct TailStats {
  long long max_work;   // K-blocks of the busiest pair
  int max_segs;         // most partial tiles held by one pair
  int nslots;           // slots used (pair level)
  long long nsegs;      // segments in all
  bool complete;        // every (tile, K-block) of the tail is assigned
  int levels;           // levels walked
};
TailStats grad_tail_stats(int G, int ntail, long long L, uint32_t cover);
// Writes the tail schedule's segments and contributions (see
// dpclip_grad_tail_schedule).
void grad_tail_dump(int G, int ntail, long long L, uint32_t cover, int64_t* segs, int seg_cap,
                    int* nsegs, int64_t* contrib, int contrib_cap, int* ncontrib);
constexpr int kMaxPersistentGrid = 160;   // CTAs of the persistent kernels (<= SMs)
size_t ghost_smem();
// Units of the ghost kernel's last round that may share a stored X: at most
// one sub-unit per pair, so at most half the largest grid of pairs.
constexpr int kGhostSharedUnits = kMaxPersistentGrid / 4;
// Tail split of the ghost units for a grid: sets nfull, tail_split,
// pb_per_split and tail_shared.
void plan_ghost_schedule(GhostParams& p, int grid);

}  // namespace dpclip
