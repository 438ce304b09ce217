// Hutch++ middle step ("Core mechanism", item 2 of the randomized-clipping
// summary: a QR-based low-rank head plus a Hutchinson tail):
//   V = O_i S (p x r, fp32, from the first two sweeps)
//   Q = orthonormal basis of range(V)        -- pivoted CholeskyQR2
//   W = G' - Q (Q^T G')                      -- tail probes projected off Q
//   out = [Q | 0 | W | 0] padded to 32 columns ([B][32][p], hi/lo bf16 for
//         the tensor-core sweep, or fp32)
// The estimate depends on Q only through span(Q) (the head is trace(Q^T O Q)
// and the tail uses I - Q Q^T), so any orthonormal basis of the same span
// gives the same result as a Householder QR.
//
// CholeskyQR2: Gram H = V^T V, Cholesky H = R^T R, Q1 = V R^-1, then once more
// on Q1 (whose Gram is close to the identity).  Everything runs in fp32: this
// GPU's fp64 pipe is a small fraction of its fp32 rate.  The first Cholesky is
// pivoted and stops at pivots below 1e-5 of the largest diagonal entry (a
// singular-value ratio of ~3e-3): such directions carry almost no energy of
// O_i (T < r makes rank(O_i) < r, for instance), so Q keeps fewer columns and
// the tail estimates the rest.  With them dropped the kept Gram has condition
// number below ~1e5, within fp32 Cholesky's reach, and the second pass
// restores orthogonality to fp32 level.
//
// Parallel layout: a cooperative grid of B x ceil(p / 512) CTAs; each CTA
// keeps its 512 rows of V (then Q) and G' in shared memory for the whole
// kernel.  Each of the three p-long reductions (V^T V, Q1^T Q1, Q^T G') writes
// one partial per CTA; after a grid-wide barrier every CTA of the sample adds
// the partials of its sample in the same fixed order, so all of them hold the
// same bits and factorise identically (one warp, lane j owns column j).
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"

namespace dpclip {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kRows = 512;           // rows of p per CTA
constexpr int kMaxR = 16;            // r = floor(k/3) <= 16 for k <= 48
constexpr int kMaxM = 18;            // m = k - 2r <= 18 for k <= 48
constexpr int kMaxE = kMaxR * kMaxM; // entries of the largest cross product
constexpr float kDropTol = 1e-5f;

struct Smem {
  float x[kMaxR][kRows + 1];       // rows of V, then Q1, then Q
  float g[kMaxM][kRows + 1];       // rows of G'
  float H[kMaxE];                  // summed cross products, row-major
  float Aw[kMaxR][kMaxR + 1];      // Cholesky workspace
  float R[kMaxR][kMaxR + 1];
  float Rinv[kMaxR][kMaxR + 1];
  int perm[kMaxR];
  int rank;
};

__device__ __forceinline__ void sym_entry(int e, int n, int& a, int& b) {
  int rem = e, row = 0, len = n;
  while (rem >= len) {
    rem -= len;
    ++row;
    --len;
  }
  a = row;
  b = row + rem;
}

// This CTA's part of X^T Y over its rows, for a < na, b < nb (upper triangle
// when sym), written to part[e].
__device__ void partial_cross(const float (*X)[kRows + 1], int na, const float (*Y)[kRows + 1],
                              int nb, bool sym, float* part) {
  const int ne = sym ? na * (na + 1) / 2 : na * nb;
  for (int e = threadIdx.x; e < ne; e += kThreads) {
    int a, b;
    if (sym) {
      sym_entry(e, na, a, b);
    } else {
      a = e / nb;
      b = e % nb;
    }
    const float* xa = X[a];
    const float* yb = Y[b];
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int c = 0; c < kRows; c += 4) {
      s0 = fmaf(xa[c], yb[c], s0);
      s1 = fmaf(xa[c + 1], yb[c + 1], s1);
      s2 = fmaf(xa[c + 2], yb[c + 2], s2);
      s3 = fmaf(xa[c + 3], yb[c + 3], s3);
    }
    part[e] = (s0 + s1) + (s2 + s3);
  }
}

// Sums the per-CTA partials of this sample (chunk order) into sm.H, expanding
// the upper triangle when sym.
__device__ void sum_partials(Smem& sm, const float* parts, int cps, int na, int nb, bool sym) {
  const int ne = sym ? na * (na + 1) / 2 : na * nb;
  for (int e = threadIdx.x; e < ne; e += kThreads) {
    float s = 0.f;
    for (int q0 = 0; q0 < cps; q0 += 8) {   // 8 loads in flight, added in chunk order
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = q0 + u < cps ? __ldcg(parts + (size_t)(q0 + u) * kMaxE + e) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    if (sym) {
      int a, b;
      sym_entry(e, na, a, b);
      sm.H[a * nb + b] = s;
      sm.H[b * nb + a] = s;
    } else {
      sm.H[e] = s;
    }
  }
}

// One warp: Cholesky of the n x n Gram in sm.H (row-major, leading dim n),
// optionally with symmetric pivoting and a relative drop tolerance.  Leaves
// sm.perm, sm.rank and Rinv = R^-1 (upper triangular, rank x rank).
__device__ void warp_cholesky_inverse(Smem& sm, int n, bool pivot) {
  const int lane = threadIdx.x & 31;
  for (int idx = lane; idx < kMaxR * kMaxR; idx += 32) {
    const int a = idx / kMaxR, b = idx % kMaxR;
    sm.Aw[a][b] = (a < n && b < n) ? sm.H[a * n + b] : 0.f;
    sm.R[a][b] = 0.f;
    sm.Rinv[a][b] = 0.f;
  }
  if (lane < kMaxR) sm.perm[lane] = lane;
  __syncwarp();
  float dmax = 0.f;
  for (int a = 0; a < n; ++a) dmax = fmaxf(dmax, sm.Aw[a][a]);
  const float tol = pivot ? kDropTol * dmax : 0.f;
  int rank = 0;
  for (int kk = 0; kk < n; ++kk) {
    int piv = kk;
    if (pivot)
      for (int j = kk + 1; j < n; ++j)
        if (sm.Aw[j][j] > sm.Aw[piv][piv]) piv = j;
    if (!(sm.Aw[piv][piv] > tol) || !(dmax > 0.f)) break;
    if (piv != kk) {
      // swap rows and columns kk <-> piv of the working matrix, the columns of
      // the finished rows of R, and the permutation
      if (lane < n) {
        const float t0 = sm.Aw[kk][lane];
        sm.Aw[kk][lane] = sm.Aw[piv][lane];
        sm.Aw[piv][lane] = t0;
      }
      __syncwarp();
      if (lane < n) {
        const float t0 = sm.Aw[lane][kk];
        sm.Aw[lane][kk] = sm.Aw[lane][piv];
        sm.Aw[lane][piv] = t0;
      }
      if (lane < kk) {
        const float t0 = sm.R[lane][kk];
        sm.R[lane][kk] = sm.R[lane][piv];
        sm.R[lane][piv] = t0;
      }
      if (lane == 0) {
        const int tp = sm.perm[kk];
        sm.perm[kk] = sm.perm[piv];
        sm.perm[piv] = tp;
      }
      __syncwarp();
    }
    const float rkk = sqrtf(sm.Aw[kk][kk]);
    if (lane >= kk && lane < n) sm.R[kk][lane] = lane == kk ? rkk : sm.Aw[kk][lane] / rkk;
    __syncwarp();
    // trailing update: Aw[a][b] -= R[kk][a] R[kk][b] for a, b > kk
    for (int idx = lane; idx < kMaxR * kMaxR; idx += 32) {
      const int a = idx / kMaxR, b = idx % kMaxR;
      if (a > kk && b > kk && a < n && b < n) sm.Aw[a][b] -= sm.R[kk][a] * sm.R[kk][b];
    }
    __syncwarp();
    ++rank;
  }
  // R^-1 by back substitution, one column per lane
  if (lane < rank) {
    const int j = lane;
    sm.Rinv[j][j] = 1.f / sm.R[j][j];
    for (int a = j - 1; a >= 0; --a) {
      float s = 0.f;
      for (int l = a + 1; l <= j; ++l) s = fmaf(sm.R[a][l], sm.Rinv[l][j], s);
      sm.Rinv[a][j] = -s / sm.R[a][a];
    }
  }
  if (lane == 0) sm.rank = rank;
  __syncwarp();
}

// In place on the shared rows: x[:, b] <- sum_{a <= b} x[:, perm[a]] Rinv[a][b]
// for b < rank, zero beyond.  Thread t owns rows t, t + 256.
__device__ void apply_rinv(Smem& sm, int ncols) {
  const int rank = sm.rank;
  for (int c = threadIdx.x; c < kRows; c += kThreads) {
    float v[kMaxR];
#pragma unroll
    for (int a = 0; a < kMaxR; ++a) v[a] = (a < rank && a < ncols) ? sm.x[sm.perm[a]][c] : 0.f;
#pragma unroll
    for (int b = 0; b < kMaxR; ++b) {
      float s = 0.f;
#pragma unroll
      for (int a = 0; a <= b; ++a) s = fmaf(v[a], sm.Rinv[a][b], s);
      sm.x[b][c] = b < rank ? s : 0.f;
    }
  }
}

__global__ void __launch_bounds__(kThreads) hpp_qr_kernel(const __grid_constant__ HppQrParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  cg::grid_group grid = cg::this_grid();
  pdl_trigger();
  pdl_wait();
  const int cps = p.cps;
  const int i = p.sample0 + (int)blockIdx.x / cps;
  const int chunk = (int)blockIdx.x % cps;
  const int c0 = chunk * kRows;
  const int r = p.r, m = p.m;
  const bool active = i < p.B;   // grids are whole samples; guard anyway
  float* part1 = p.part + ((size_t)0 * p.B + (active ? i : 0)) * cps * kMaxE;
  float* part2 = p.part + ((size_t)1 * p.B + (active ? i : 0)) * cps * kMaxE;
  float* part3 = p.part + ((size_t)2 * p.B + (active ? i : 0)) * cps * kMaxE;

  // ---- stage this CTA's rows of V (r columns) and G' (m columns); the loads
  // of 16 consecutive elements per thread are issued before any is stored
  constexpr int kBatch = 16;
  for (int it0 = 0; it0 < kMaxR * kRows; it0 += kBatch * kThreads) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int idx = it0 + u * kThreads + threadIdx.x;
      const int a = idx / kRows, c = idx % kRows;
      v[u] = (active && a < r && c0 + c < p.p) ? p.V[((size_t)i * p.ldv + a) * p.p + c0 + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int idx = it0 + u * kThreads + threadIdx.x;
      sm.x[idx / kRows][idx % kRows] = v[u];
    }
  }
  for (int it0 = 0; it0 < kMaxM * kRows; it0 += kBatch * kThreads) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int idx = it0 + u * kThreads + threadIdx.x;
      const int l = idx / kRows, c = idx % kRows;
      float x = 0.f;
      if (idx < kMaxM * kRows && active && l < m && c0 + c < p.p) {
        const size_t o = (size_t)l * p.p + c0 + c;
        x = p.gp_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.Gp)[o])
                      : static_cast<const float*>(p.Gp)[o];
      }
      v[u] = x;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int idx = it0 + u * kThreads + threadIdx.x;
      if (idx < kMaxM * kRows) sm.g[idx / kRows][idx % kRows] = v[u];
    }
  }
  __syncthreads();

  // ---- pass 1: pivoted Cholesky of V^T V; Q1 = V P R^-1
  if (active) partial_cross(sm.x, r, sm.x, r, true, part1 + (size_t)chunk * kMaxE);
  __threadfence();
  grid.sync();
  if (active) sum_partials(sm, part1, cps, r, r, true);
  __syncthreads();
  if (threadIdx.x < 32) warp_cholesky_inverse(sm, r, true);
  __syncthreads();
  apply_rinv(sm, r);
  __syncthreads();
  const int rank1 = sm.rank;

  // ---- pass 2: Cholesky of Q1^T Q1 (close to the identity); Q = Q1 R2^-1
  if (active) partial_cross(sm.x, rank1, sm.x, rank1, true, part2 + (size_t)chunk * kMaxE);
  __threadfence();
  grid.sync();
  if (active) sum_partials(sm, part2, cps, rank1, rank1, true);
  __syncthreads();
  if (threadIdx.x < 32) warp_cholesky_inverse(sm, rank1, false);
  __syncthreads();
  apply_rinv(sm, rank1);
  __syncthreads();
  const int rank = sm.rank;

  // ---- tail probes: C = Q^T G' (rank x m), W = G' - Q C
  if (active) partial_cross(sm.x, rank, sm.g, m, false, part3 + (size_t)chunk * kMaxE);
  __threadfence();
  grid.sync();
  if (active) sum_partials(sm, part3, cps, rank, m, false);
  __syncthreads();
  if (!active) return;
  for (int idx = threadIdx.x; idx < kMaxNP * kRows; idx += kThreads) {
    const int j = idx / kRows, c = idx % kRows;
    if (c0 + c >= p.p) continue;
    float val = 0.f;
    if (j < rank) {
      val = sm.x[j][c];
    } else if (j >= r && j < r + m) {
      const int l = j - r;
      float s = sm.g[l][c];
      for (int a = 0; a < rank; ++a) s = fmaf(-sm.x[a][c], sm.H[a * m + l], s);
      val = s;
    }
    const size_t o = ((size_t)i * kMaxNP + j) * p.p + c0 + c;
    if (p.out_f32) {
      p.out_f32[o] = val;
    } else {
      __nv_bfloat16 hi, lo;
      split_hilo(val, hi, lo);
      p.out_hi[o] = hi;
      p.out_lo[o] = lo;
    }
  }
}

}  // namespace

size_t hpp_qr_part_floats(int B, int p) { return (size_t)3 * B * ((p + kRows - 1) / kRows) * kMaxE; }

cudaError_t launch_hpp_qr(const HppQrParams& p_in, cudaStream_t s) {
  if (p_in.r > kMaxR || p_in.m > kMaxM || p_in.r + p_in.m > kMaxNP) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Smem);
  cudaError_t e =
      cudaFuncSetAttribute(hpp_qr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hpp_qr_kernel, kThreads, smem)) !=
      cudaSuccess)
    return e;
  HppQrParams p = p_in;
  p.cps = (p.p + kRows - 1) / kRows;
  const int resident = std::max(1, per_sm * nsm);
  if (p.cps > resident) return cudaErrorCooperativeLaunchTooLarge;
  // whole samples per cooperative launch, as many as stay co-resident
  const int per_launch = std::max(1, resident / p.cps);
  for (int s0 = 0; s0 < p.B; s0 += per_launch) {
    p.sample0 = s0;
    const int nb = std::min(per_launch, p.B - s0);
    e = launch_pdl(hpp_qr_kernel, dim3(nb * p.cps), dim3(kThreads), smem, s, true, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dpclip
