// Hutch++ middle step ("Core mechanism", item 2 of the randomized-clipping
// summary: a QR-based low-rank head plus a Hutchinson tail):
//   V = O_i S (p x r, fp32, from the first two sweeps)
//   Q = orthonormal basis of range(V)        -- CholeskyQR2 with column drop
//   W = G' - Q (Q^T G')                      -- tail probes projected off Q
//   out = [Q | 0 | W | 0] padded to 32 columns ([B][32][p], hi/lo bf16 for
//         the tensor-core sweep, or fp32)
// The estimate depends on Q only through span(Q) (the head is trace(Q^T O Q)
// and the tail uses I - Q Q^T), so any orthonormal basis of the same span
// gives the same result as a Householder QR.
//
// CholeskyQR2: Gram H = V^T V, Cholesky H = R^T R, Q1 = V R^-1, then once more
// on Q1 (whose Gram is close to the identity).  Everything runs in fp32: this
// GPU's fp64 pipe is a small fraction of its fp32 rate.  A Cholesky pivot
// below 1e-5 of the largest diagonal entry (a singular-value ratio of ~3e-3)
// marks its column as dependent on the earlier ones: that column of Q is set
// to zero, so Q spans the rest and the tail estimates what is left (T < r
// makes rank(O_i) < r, for instance).  With those columns dropped the kept
// Gram has condition number below ~1e5, within fp32 Cholesky's reach, and the
// second pass restores orthogonality to fp32 level.
//
// Parallel layout: a cooperative grid of B x ceil(p / 512) CTAs; each CTA
// keeps its 512 rows of V (then Q) and G' in shared memory for the whole
// kernel.  Two p-long reductions: V^T V, then Q1^T Q1 together with
// Q1^T G' (Q^T G' = R2^-T Q1^T G' needs no third pass).  Each writes one
// partial per CTA; after a grid-wide barrier every CTA of the sample adds the
// partials of its sample in the same fixed order, so all of them hold the
// same bits and factorise identically (one thread, the r x r factor fully in
// registers; rows apply R^-1 by forward substitution).
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
constexpr int kSym = kMaxR * (kMaxR + 1) / 2;     // 136 upper-triangle entries
constexpr int kPartStride = 512;     // floats per CTA partial
static_assert(kSym + kMaxR * kMaxM <= kPartStride, "partials of pass 2 must fit");
constexpr float kDropTol = 1e-5f;

struct Smem {
  float x[kMaxR][kRows + 1];       // rows of V, then Q1, then Q
  float g[kMaxM][kRows + 1];       // rows of G'
  float S[kPartStride];            // summed partials of the current pass
  float H[kMaxR][kMaxR + 1];       // Gram matrix of the current pass
  float K[kMaxR][kMaxM];           // Q1^T G'
  float Cm[kMaxR][kMaxM];          // Q^T G' = R2^-T K (zero rows for dropped columns)
  float R[kMaxR][kMaxR + 1];       // Cholesky factor (zero rows for dropped columns)
  float rdiag[kMaxR];              // 1 / R[k][k], or 0 for a dropped column
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

// sm.S[e] = sum of the per-CTA partials of this sample (chunk order), e < ne.
__device__ void sum_partials(Smem& sm, const float* parts, int cps, int ne) {
  for (int e = threadIdx.x; e < ne; e += kThreads) {
    float s = 0.f;
    for (int q0 = 0; q0 < cps; q0 += 8) {   // 8 loads in flight, added in chunk order
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = q0 + u < cps ? __ldcg(parts + (size_t)(q0 + u) * kPartStride + e) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    sm.S[e] = s;
  }
}

// sm.H (n x n) from the upper-triangle sums in sm.S[0 .. n(n+1)/2).
__device__ void expand_sym(Smem& sm, int n) {
  for (int e = threadIdx.x; e < n * (n + 1) / 2; e += kThreads) {
    int a, b;
    sym_entry(e, n, a, b);
    sm.H[a][b] = sm.S[e];
    sm.H[b][a] = sm.S[e];
  }
}

// One thread: Cholesky H = R^T R of the n x n Gram in sm.H, fully unrolled in
// registers.  A pivot below kDropTol times the largest diagonal entry marks
// its column as dependent on the earlier ones: its row of R and its entry of
// rdiag (= 1 / R[k][k]) are zero, so the matching column of Q comes out zero
// and drops out of both the head and the tail projection.
__device__ void serial_cholesky(Smem& sm, int n) {
  float a[kMaxR][kMaxR];
#pragma unroll
  for (int i = 0; i < kMaxR; ++i)
#pragma unroll
    for (int j = i; j < kMaxR; ++j) a[i][j] = (i < n && j < n) ? sm.H[i][j] : 0.f;
  float dmax = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) dmax = fmaxf(dmax, a[i][i]);
  const float tol = kDropTol * dmax;
#pragma unroll
  for (int k = 0; k < kMaxR; ++k) {
    const bool keep = k < n && a[k][k] > tol && dmax > 0.f;
    const float rkk = keep ? sqrtf(a[k][k]) : 0.f;
    const float inv = keep ? 1.f / rkk : 0.f;
    sm.rdiag[k] = inv;
    a[k][k] = rkk;
#pragma unroll
    for (int j = k + 1; j < kMaxR; ++j) a[k][j] *= inv;
#pragma unroll
    for (int i = k + 1; i < kMaxR; ++i)
#pragma unroll
      for (int j = i; j < kMaxR; ++j) a[i][j] = fmaf(-a[k][i], a[k][j], a[i][j]);
  }
#pragma unroll
  for (int i = 0; i < kMaxR; ++i)
#pragma unroll
    for (int j = 0; j < kMaxR; ++j) sm.R[i][j] = j >= i ? a[i][j] : 0.f;
}

// In place on the shared rows: x[c, :] <- x[c, :] R^-1 by forward
// substitution, q[b] = (x[b] - sum_{a<b} q[a] R[a][b]) / R[b][b] (zero for a
// dropped column).  Thread t owns rows t, t + 256.
__device__ void apply_rinv(Smem& sm, int n) {
  for (int c = threadIdx.x; c < kRows; c += kThreads) {
    float q[kMaxR];
#pragma unroll
    for (int b = 0; b < kMaxR; ++b) {
      float s = b < n ? sm.x[b][c] : 0.f;
#pragma unroll
      for (int a = 0; a < b; ++a) s = fmaf(-q[a], sm.R[a][b], s);
      q[b] = s * sm.rdiag[b];
    }
#pragma unroll
    for (int b = 0; b < kMaxR; ++b) sm.x[b][c] = q[b];
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
  const int ia = active ? i : 0;
  float* part1 = p.part + ((size_t)0 * p.B + ia) * cps * kPartStride;
  float* part2 = p.part + ((size_t)1 * p.B + ia) * cps * kPartStride;

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

  // ---- pass 1: Cholesky of V^T V; Q1 = V R1^-1
  const int ne = r * (r + 1) / 2;
  if (active) partial_cross(sm.x, r, sm.x, r, true, part1 + (size_t)chunk * kPartStride);
  __threadfence();
  grid.sync();
  if (active) sum_partials(sm, part1, cps, ne);
  __syncthreads();
  expand_sym(sm, r);
  __syncthreads();
  if (threadIdx.x == 0) serial_cholesky(sm, r);
  __syncthreads();
  apply_rinv(sm, r);
  __syncthreads();

  // ---- pass 2, one reduction for both: Q1^T Q1 (close to the identity) and
  // K = Q1^T G'.  Then Q = Q1 R2^-1 and Q^T G' = R2^-T K.
  if (active) {
    float* mine = part2 + (size_t)chunk * kPartStride;
    partial_cross(sm.x, r, sm.x, r, true, mine);
    partial_cross(sm.x, r, sm.g, m, false, mine + ne);
  }
  __threadfence();
  grid.sync();
  if (active) sum_partials(sm, part2, cps, ne + r * m);
  __syncthreads();
  expand_sym(sm, r);
  for (int e = threadIdx.x; e < r * m; e += kThreads) sm.K[e / m][e % m] = sm.S[ne + e];
  __syncthreads();
  if (threadIdx.x == 0) serial_cholesky(sm, r);
  __syncthreads();
  // C = R2^-T K by forward substitution, one tail column per thread
  if (threadIdx.x < m) {
    const int l = threadIdx.x;
    float cc[kMaxR];
#pragma unroll
    for (int b = 0; b < kMaxR; ++b) {
      float s = b < r ? sm.K[b][l] : 0.f;
#pragma unroll
      for (int a = 0; a < b; ++a) s = fmaf(-sm.R[a][b], cc[a], s);
      cc[b] = s * sm.rdiag[b];
      sm.Cm[b][l] = cc[b];
    }
  }
  apply_rinv(sm, r);
  __syncthreads();
  if (!active) return;

  // ---- outputs [Q | W | 0], W = G' - Q (Q^T G'); each thread owns rows
  for (int c = threadIdx.x; c < kRows; c += kThreads) {
    if (c0 + c >= p.p) break;
    float qrow[kMaxR];
#pragma unroll
    for (int a = 0; a < kMaxR; ++a) qrow[a] = sm.x[a][c];
#pragma unroll
    for (int j = 0; j < kMaxNP; ++j) {
      float val = 0.f;
      if (j < kMaxR && j < r) {
        val = qrow[j < kMaxR ? j : 0];
      } else if (j >= r && j < r + m) {
        const int l = j - r;
        float s = sm.g[l][c];
#pragma unroll
        for (int a = 0; a < kMaxR; ++a) s = fmaf(-qrow[a], sm.Cm[a][l], s);
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
}

}  // namespace

size_t hpp_qr_part_floats(int B, int p) {
  return (size_t)2 * B * ((p + kRows - 1) / kRows) * kPartStride;
}

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
