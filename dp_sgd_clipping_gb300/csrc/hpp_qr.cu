// Hutch++ middle step ("Core mechanism", item 2 of the randomized-clipping
// summary: a QR-based low-rank head plus a Hutchinson tail), one CTA per
// sample:
//   V = O_i S (p x r, fp32, from the first two sweeps)
//   Q = orthonormal basis of range(V)        -- pivoted CholeskyQR2 in fp64
//   W = G' - Q (Q^T G')                      -- tail probes projected off Q
//   out = [Q | 0 | W | 0] padded to 32 columns ([B][32][p], hi/lo bf16 for
//         the tensor-core sweep, or fp32)
// The estimate depends on Q only through span(Q) (the head is trace(Q^T O Q)
// and the tail uses I - Q Q^T), so any orthonormal basis of the same span
// gives the same result as a Householder QR.  CholeskyQR2: Gram H = V^T V in
// fp64, Cholesky H = R^T R, Q1 = V R^-1, then once more on Q1.  The first
// Cholesky is pivoted and stops at pivots below 1e-7 of the largest diagonal
// entry: those directions carry no energy of O_i beyond rounding noise (e.g.
// T < r makes rank(O_i) < r), so Q keeps fewer columns and the tail covers the
// rest.
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kThreads = 512;
constexpr int kChunk = 256;          // rows of p staged in shared memory per pass
constexpr int kMaxR = 16;            // r = floor(k/3) <= 16 for k <= 48
constexpr int kMaxM = 18;            // m = k - 2r <= 18 for k <= 48
constexpr double kDropTol = 1e-7;

enum SrcType { kF32 = 0, kF64 = 1, kBF16 = 2 };
struct Src {
  const void* ptr;
  int type;
  long long ld;   // element stride between rows (columns of the p x n matrix)
};

__device__ __forceinline__ double src_at(const Src& s, int a, int c) {
  const long long idx = (long long)a * s.ld + c;
  if (s.type == kF32) return (double)static_cast<const float*>(s.ptr)[idx];
  if (s.type == kF64) return static_cast<const double*>(s.ptr)[idx];
  return (double)__bfloat162float(static_cast<const __nv_bfloat16*>(s.ptr)[idx]);
}

struct Smem {
  double x[kMaxR][kChunk + 1];
  double y[kMaxM][kChunk + 1];
  double red[kThreads];
  double H[kMaxR * kMaxM];
  double R[kMaxR][kMaxR];
  double Rinv[kMaxR][kMaxR];
  int perm[kMaxR];
  int rank;
};

// out[a * nb + b] = sum_{c < p} X(a, c) Y(b, c) in fp64, for a < na, b < nb
// (b >= a only when sym).  Deterministic: fixed row partition, fixed order.
__device__ void cross_products(Smem& sm, const Src& X, int na, const Src& Y, int nb, bool sym,
                               int p, double* out) {
  const int ne = sym ? na * (na + 1) / 2 : na * nb;
  if (ne == 0) return;
  const int groups = kThreads / ne;
  const int t = threadIdx.x;
  int ea = 0, eb = 0, g = -1;
  if (t < ne * groups) {
    const int e = t % ne;
    g = t / ne;
    if (sym) {
      int rem = e, a = 0, len = na;
      while (rem >= len) {
        rem -= len;
        ++a;
        --len;
      }
      ea = a;
      eb = a + rem;
    } else {
      ea = e / nb;
      eb = e % nb;
    }
  }
  double acc = 0.0;
  for (int c0 = 0; c0 < p; c0 += kChunk) {
    const int n = min(kChunk, p - c0);
    __syncthreads();
    for (int idx = t; idx < na * n; idx += kThreads) {
      const int a = idx / n, c = idx % n;
      sm.x[a][c] = src_at(X, a, c0 + c);
    }
    if (!sym) {
      for (int idx = t; idx < nb * n; idx += kThreads) {
        const int b = idx / n, c = idx % n;
        sm.y[b][c] = src_at(Y, b, c0 + c);
      }
    }
    __syncthreads();
    if (g >= 0) {
      const double* xa = sm.x[ea];
      const double* yb = sym ? sm.x[eb] : sm.y[eb];
      for (int c = g; c < n; c += groups) acc = fma(xa[c], yb[c], acc);
    }
  }
  __syncthreads();
  sm.red[t] = acc;
  __syncthreads();
  if (t < ne) {
    double s = 0.0;
    for (int gg = 0; gg < groups; ++gg) s += sm.red[gg * ne + t];
    int a = 0, b = 0;
    if (sym) {
      int rem = t, len = na;
      while (rem >= len) {
        rem -= len;
        ++a;
        --len;
      }
      b = a + rem;
      out[a * nb + b] = s;
      out[b * nb + a] = s;
    } else {
      a = t / nb;
      b = t % nb;
      out[a * nb + b] = s;
    }
  }
  __syncthreads();
}

// Upper-triangular inverse of the leading n x n block of R.
__device__ void upper_inverse(const double (&R)[kMaxR][kMaxR], double (&Ri)[kMaxR][kMaxR], int n) {
  for (int a = 0; a < kMaxR; ++a)
    for (int b = 0; b < kMaxR; ++b) Ri[a][b] = 0.0;
  for (int j = 0; j < n; ++j) {
    Ri[j][j] = 1.0 / R[j][j];
    for (int a = j - 1; a >= 0; --a) {
      double s = 0.0;
      for (int l = a + 1; l <= j; ++l) s += R[a][l] * Ri[l][j];
      Ri[a][j] = -s / R[a][a];
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) hpp_qr_kernel(const __grid_constant__ HppQrParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int i = blockIdx.x;
  const int r = p.r, m = p.m;
  const Src V{p.V + (size_t)i * p.ldv * p.p, kF32, p.p};
  double* Q1 = p.Q1 + (size_t)i * r * p.p;
  const Src Q1s{Q1, kF64, p.p};
  const Src Gp{p.Gp, p.gp_bf16 ? kBF16 : kF32, p.p};

  // ---- pass 1: pivoted Cholesky of V^T V
  cross_products(sm, V, r, V, r, true, p.p, sm.H);
  if (threadIdx.x == 0) {
    double Aw[kMaxR][kMaxR];
    for (int a = 0; a < r; ++a) {
      sm.perm[a] = a;
      for (int b = 0; b < r; ++b) Aw[a][b] = sm.H[a * r + b];
    }
    double dmax = 0.0;
    for (int a = 0; a < r; ++a) dmax = fmax(dmax, Aw[a][a]);
    const double tol = kDropTol * dmax;
    for (int a = 0; a < kMaxR; ++a)
      for (int b = 0; b < kMaxR; ++b) sm.R[a][b] = 0.0;
    int rank = 0;
    for (int kk = 0; kk < r; ++kk) {
      int piv = kk;
      for (int j = kk + 1; j < r; ++j)
        if (Aw[j][j] > Aw[piv][piv]) piv = j;
      if (!(Aw[piv][piv] > tol) || dmax <= 0.0) break;
      if (piv != kk) {
        for (int j = 0; j < r; ++j) {
          const double t0 = Aw[kk][j];
          Aw[kk][j] = Aw[piv][j];
          Aw[piv][j] = t0;
        }
        for (int j = 0; j < r; ++j) {
          const double t0 = Aw[j][kk];
          Aw[j][kk] = Aw[j][piv];
          Aw[j][piv] = t0;
        }
        for (int j = 0; j < kk; ++j) {
          const double t0 = sm.R[j][kk];
          sm.R[j][kk] = sm.R[j][piv];
          sm.R[j][piv] = t0;
        }
        const int tp = sm.perm[kk];
        sm.perm[kk] = sm.perm[piv];
        sm.perm[piv] = tp;
      }
      const double rkk = sqrt(Aw[kk][kk]);
      sm.R[kk][kk] = rkk;
      for (int j = kk + 1; j < r; ++j) sm.R[kk][j] = Aw[kk][j] / rkk;
      for (int a = kk + 1; a < r; ++a)
        for (int b = kk + 1; b < r; ++b) Aw[a][b] -= sm.R[kk][a] * sm.R[kk][b];
      ++rank;
    }
    sm.rank = rank;
    upper_inverse(sm.R, sm.Rinv, rank);
  }
  __syncthreads();
  int rank = sm.rank;

  // Q1 = V[:, perm[:rank]] R^-1, rows distributed over the threads
  for (int c = threadIdx.x; c < p.p; c += kThreads) {
    double v[kMaxR];
    for (int a = 0; a < rank; ++a) v[a] = src_at(V, sm.perm[a], c);
    for (int b = 0; b < rank; ++b) {
      double s = 0.0;
      for (int a = 0; a <= b; ++a) s = fma(v[a], sm.Rinv[a][b], s);
      Q1[(size_t)b * p.p + c] = s;
    }
  }
  __syncthreads();

  // ---- pass 2: plain Cholesky of Q1^T Q1 (close to the identity)
  cross_products(sm, Q1s, rank, Q1s, rank, true, p.p, sm.H);
  if (threadIdx.x == 0) {
    double Aw[kMaxR][kMaxR];
    for (int a = 0; a < rank; ++a)
      for (int b = 0; b < rank; ++b) Aw[a][b] = sm.H[a * rank + b];
    for (int a = 0; a < kMaxR; ++a)
      for (int b = 0; b < kMaxR; ++b) sm.R[a][b] = 0.0;
    int rank2 = 0;
    for (int kk = 0; kk < rank; ++kk) {
      if (!(Aw[kk][kk] > 0.0)) break;
      const double rkk = sqrt(Aw[kk][kk]);
      sm.R[kk][kk] = rkk;
      for (int j = kk + 1; j < rank; ++j) sm.R[kk][j] = Aw[kk][j] / rkk;
      for (int a = kk + 1; a < rank; ++a)
        for (int b = kk + 1; b < rank; ++b) Aw[a][b] -= sm.R[kk][a] * sm.R[kk][b];
      ++rank2;
    }
    sm.rank = rank2;
    upper_inverse(sm.R, sm.Rinv, rank2);
  }
  __syncthreads();
  rank = sm.rank;
  for (int c = threadIdx.x; c < p.p; c += kThreads) {
    double v[kMaxR];
    for (int a = 0; a < rank; ++a) v[a] = Q1[(size_t)a * p.p + c];
    for (int b = 0; b < rank; ++b) {
      double s = 0.0;
      for (int a = 0; a <= b; ++a) s = fma(v[a], sm.Rinv[a][b], s);
      Q1[(size_t)b * p.p + c] = s;
    }
  }
  __syncthreads();

  // ---- tail probes: C = Q^T G' (rank x m), W = G' - Q C
  cross_products(sm, Q1s, rank, Gp, m, false, p.p, sm.H);
  for (int c = threadIdx.x; c < p.p; c += kThreads) {
    double q[kMaxR];
    for (int a = 0; a < rank; ++a) q[a] = Q1[(size_t)a * p.p + c];
    for (int j = 0; j < kMaxNP; ++j) {
      double val = 0.0;
      if (j < rank) {
        val = q[j];
      } else if (j >= r && j < r + m) {
        const int l = j - r;
        double s = src_at(Gp, l, c);
        for (int a = 0; a < rank; ++a) s -= q[a] * sm.H[a * m + l];
        val = s;
      }
      const size_t o = ((size_t)i * kMaxNP + j) * p.p + c;
      if (p.out_f32) {
        p.out_f32[o] = (float)val;
      } else {
        __nv_bfloat16 hi, lo;
        split_hilo((float)val, hi, lo);
        // the fp32 rounding of val is below the hi/lo split's resolution
        p.out_hi[o] = hi;
        p.out_lo[o] = lo;
      }
    }
  }
}

}  // namespace

cudaError_t launch_hpp_qr(const HppQrParams& p, cudaStream_t s) {
  if (p.r > kMaxR || p.m > kMaxM || p.r + p.m > kMaxNP) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Smem);
  cudaError_t e =
      cudaFuncSetAttribute(hpp_qr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  hpp_qr_kernel<<<p.B, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dpclip
