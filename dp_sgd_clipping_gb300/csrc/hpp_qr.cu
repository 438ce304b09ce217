// Hutch++ middle step ("Core mechanism", item 2 of the randomized-clipping
// summary: a QR-based low-rank head plus a Hutchinson tail):
//   V = O_i S (p x r, fp32, from the first two sweeps)
//   Q = orthonormal basis of range(V)        -- CholeskyQR2 with column drop
//   W = G' - Q (Q^T G')                      -- tail probes projected off Q
//   out = [Q | W | 0] padded to 32 columns ([B][32][p], hi/lo bf16 for the
//         tensor-core sweep, or fp32)
// The estimate depends on Q only through span(Q) (the head is trace(Q^T O Q)
// and the tail uses I - Q Q^T), so any orthonormal basis of the same span
// gives the same result as a Householder QR.
//
// CholeskyQR2: Gram H = V^T V, Cholesky H = R^T R, Q1 = V R^-1, then once more
// on Q1 (whose Gram is close to the identity).  For bf16 inputs everything
// runs in fp32 (this GPU's fp64 pipe is a small fraction of its fp32 rate,
// and V itself carries only ~16 bits).  A Cholesky pivot below 1e-5 of the
// largest diagonal entry (a singular-value ratio of ~3e-3) marks its column
// as dependent on the earlier ones: that column of Q is set to zero, so Q
// spans the rest and the tail estimates what is left (T < r makes
// rank(O_i) < r, for instance).  With those columns dropped the kept Gram has
// condition number below ~1e5, within fp32 Cholesky's reach, and the second
// pass restores orthogonality to fp32 level.
//
// For fp32 inputs the first pass's Gram, its Cholesky factor and R^-1 are
// formed in fp64 (the fp32 products are exact in fp64), and only pivots
// below 1e-12 of the largest are dropped: the squared singular values of
// O_i S fall as the fourth power of those of A_i^T G_i, so on a decaying
// spectrum the fp32 rule would hand most of the head's directions to the
// tail, whose estimate then differs from an exact QR's by far more than
// fp32 rounding.  Q1 = V R^-1 is still formed in fp32; its loss of
// orthogonality (about the fp32 unit roundoff times the condition number of
// V) is what the second, fp32 pass removes.
//
// Parallel layout: one thread-block cluster per sample (up to 16 CTAs where
// the device allows clusters that large, else 8; fewer for short p).  CTA j
// of the cluster owns a contiguous range of rows of V and G', staged in its
// shared memory column by column ([x (r) | g (m)] columns, rows contiguous)
// by 16-byte asynchronous copies (one round trip to L2).  The two p-long
// reductions, V^T V and then Q1^T [Q1 | G'] (which also gives
// Q^T G' = R2^-T Q1^T G' without a third pass), run as register-blocked
// 4 x 4 outer products per thread; each CTA publishes its partial in its own
// shared memory and, after a cluster barrier, every CTA reads the partials
// of all ranks through distributed shared memory and adds them in rank
// order.  All CTAs of the sample thus hold the same bits and factorise
// identically.  R^-1 is then formed once as a small matrix M (the forward
// substitution applied to unit rows), and rows are transformed as x M.  No
// global scratch, no grid-wide barrier.
//
// Latency, not arithmetic, sets this kernel's time: every phase runs once
// per CTA, so the first fetch of each phase's instructions is on the
// critical path.  The factorisation (lane-parallel, in registers) and the
// unrolled inverse are non-inlined functions that a spare warp runs once on
// scratch while the first tile's copies are in flight; every other function
// has a single call site.
#include <cooperative_groups.h>

#include <algorithm>

#include <atomic>

#include "common.cuh"

namespace dpclip {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kTileRows = 512;       // rows resident per CTA (more: tiles re-staged)
constexpr int kRowsTarget = 512;     // rows per CTA the cluster size aims at
constexpr int kLdc = kTileRows + 4;  // floats per staged column (16-byte aligned)
constexpr int kCols = 32;            // staged columns: [x (r) | g (m)], r + m <= 32
constexpr int kMaxR = 16;            // r = floor(k/3) <= 16 for k <= 48
constexpr int kMaxM = 18;            // m = k - 2r <= 18 for k <= 48
constexpr int kPub = kMaxR * kMaxNP; // one CTA's partial: r x (r + m) <= 16 x 32
constexpr float kDropTol = 1e-5f;
constexpr double kDropTol64 = 1e-12;

struct Smem {
  float xs[kCols][kLdc];           // staged columns: V (then Q1, then Q) | G'
  __nv_bfloat16 gtmp[kMaxM][kTileRows];   // bf16 G' as copied, before widening
  float red[kThreads * 16];        // per-thread 4 x 4 partial blocks
  float pub[2][kPub];              // this CTA's partials of pass 1 and 2 (read by the cluster)
  float sum[kPub];                 // cluster sum of the current pass
  float K[kMaxR][kMaxM];           // Q1^T G'
  float CmT[kMaxM][kMaxR];         // (Q^T G')^T = (R2^-T K)^T, zero for columns >= r
  float R1[kMaxR][kMaxR + 1];      // Gram, then its Cholesky factor (upper triangle)
  float R2[kMaxR][kMaxR + 1];
  float rd1[kMaxR];                // 1 / R[k][k], or 0 for a dropped column
  float rd2[kMaxR];
  float M1[kMaxR][kMaxR];          // R^-1 as the forward substitution applies it
  float M2[kMaxR][kMaxR];          // (zero outside the leading r x r block)
};

// The fp64 first pass of fp32 inputs: partials, cluster sum and factor.
// Placed after Smem in dynamic shared memory, only by that instantiation.
struct Smem64 {
  double red[kThreads * 16];
  double pub[kMaxR * kMaxR];
  double sum[kMaxR * kMaxR];
  double R[kMaxR][kMaxR + 1];
  double rd[kMaxR];
};

__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
__device__ __forceinline__ double rsqrt_t(double x) { return 1.0 / sqrt(x); }

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Copies n consecutive fp32 values to shared memory: 16-byte copies when both
// ends allow it (vec), else 4-byte ones.
__device__ __forceinline__ void copy_f32(float* dst, const float* src, int n, bool vec) {
  if (vec) {
    for (int q = threadIdx.x; q < n / 4; q += kThreads) cp_async16(dst + 4 * q, src + 4 * q);
  } else {
    for (int c = threadIdx.x; c < n; c += kThreads) cp_async4(dst + c, src + c);
  }
}

// Warp 0, lane a < 16: row a of M = R^-1 as the forward substitution
// q[b] = (x[b] - sum_{a<b} q[a] R[a][b]) rdiag[b] applies it to a unit row:
// x M is that substitution for any row x (it is linear in x), and a dropped
// column b (rdiag[b] = 0) is a zero column of M.  Entries outside the
// leading r x r block are zero.  Not inlined: the two factorisations and
// the instruction-cache warm-up below run the same code.
template <typename T>
__device__ __noinline__ void invert_factor(const T (*R)[kMaxR + 1], const T* rdiag, int r,
                                           float (*M)[kMaxR]) {
  const int a = threadIdx.x & 31;
  if (a >= kMaxR) return;
  T q[kMaxR];
#pragma unroll
  for (int b = 0; b < kMaxR; ++b) {
    T s = (a == b && b < r) ? T(1) : T(0);
#pragma unroll
    for (int c = 0; c < b; ++c) s = fma(-q[c], R[c][b], s);
    q[b] = b < r ? s * rdiag[b] : T(0);
  }
#pragma unroll
  for (int b = 0; b < kMaxR; ++b) M[a][b] = a < r ? (float)q[b] : 0.f;
}

template <typename T>
__device__ __noinline__ void cholesky(T (*A)[kMaxR + 1], int n, T* rdiag, T droptol);

// Stages rows [base, base + nvalid) of V (columns < r) and G' (m columns) as
// xs[col][c], col < r + m; rows nvalid .. (nvalid rounded up to 4) are zero,
// nothing else past nvalid is read later.  Asynchronous copies throughout
// (bf16 G' as 8-element chunks, widened after they land), so the tile costs
// one round trip.  Ends with a CTA barrier.
__device__ __forceinline__ void stage_tile(Smem& sm, const HppQrParams& p, int i, int base, int nvalid,
                                           bool warm) {
  const int r = p.r, m = p.m;
  const bool vec = (p.p % 4) == 0;   // then base, nvalid and every column start are 16-byte aligned
  for (int col = 0; col < r; ++col)
    copy_f32(sm.xs[col], p.V + ((size_t)i * p.ldv + col) * p.p + base, nvalid, vec);
  if (p.gp_bf16) {
    // p % 8 == 0 on this path: base and nvalid are multiples of 8
    for (int l = 0; l < m; ++l) {
      const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.Gp) + (size_t)l * p.p + base;
      for (int q = threadIdx.x; q < nvalid / 8; q += kThreads)
        cp_async16(&sm.gtmp[l][8 * q], src + 8 * q);
    }
  } else {
    for (int l = 0; l < m; ++l)
      copy_f32(sm.xs[r + l], static_cast<const float*>(p.Gp) + (size_t)l * p.p + base, nvalid, vec);
  }
  if (warm && threadIdx.x >= 32 && threadIdx.x < 64) {
    // While the copies are in flight, warp 1 runs the (unrolled, once-per-
    // pass) factorisation and inverse on the second factor's scratch, which
    // pass 1 overwrites: that fetches their code into the instruction cache
    // before the first real use, where the fetch would otherwise sit on the
    // critical path.
    cholesky<float>(sm.R2, r, sm.rd2, kDropTol);
    invert_factor<float>(sm.R2, sm.rd2, r, sm.M2);
  }
  cp_async_wait_all();
  if (p.gp_bf16) {
    __syncthreads();
    for (int l = 0; l < m; ++l)
      for (int c = threadIdx.x; c < nvalid; c += kThreads)
        sm.xs[r + l][c] = __bfloat162float(sm.gtmp[l][c]);
  }
  const int pad = ((nvalid + 3) & ~3) - nvalid;
  for (int e = threadIdx.x; e < pad * (r + m); e += kThreads) sm.xs[e / pad][nvalid + e % pad] = 0.f;
  __syncthreads();
}

// Geometry of the register-blocked product C = X^T Y, X = columns [0, na),
// Y = columns [0, nb) of the staged tile: 4 x 4 output blocks, and the
// threads left over split the rows, in groups of 4, into `slices`
// interleaved slices.
struct Blocking {
  int nbb, nblk, slices;
  __device__ Blocking(int na, int nb) {
    nbb = (nb + 3) / 4;
    nblk = ((na + 3) / 4) * nbb;
    slices = kThreads / nblk;
  }
};

// acc += this thread's share of X^T Y over staged rows [0, nrows): block
// (a0.., b0..) over the row groups 4 (s + k slices) .. + 3.
template <typename T>
__device__ __forceinline__ void accumulate(const Smem& sm, const Blocking& bk, int nrows,
                                           T (&acc)[4][4]) {
  const int blk = (int)threadIdx.x % bk.nblk, s = (int)threadIdx.x / bk.nblk;
  if (s >= bk.slices) return;
  const int a0 = (blk / bk.nbb) * 4, b0 = (blk % bk.nbb) * 4;
  const int ngroups = (nrows + 3) / 4;
#pragma unroll 2
  for (int g = s; g < ngroups; g += bk.slices) {
    float4 x[4], y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = *reinterpret_cast<const float4*>(&sm.xs[a0 + u][4 * g]);
#pragma unroll
    for (int w = 0; w < 4; ++w) y[w] = *reinterpret_cast<const float4*>(&sm.xs[b0 + w][4 * g]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        T a = acc[u][w];
        a = fma((T)x[u].x, (T)y[w].x, a);
        a = fma((T)x[u].y, (T)y[w].y, a);
        a = fma((T)x[u].z, (T)y[w].z, a);
        a = fma((T)x[u].w, (T)y[w].w, a);
        acc[u][w] = a;
      }
  }
}

// pub[a * nb + b] = this CTA's sum of X^T Y, the slices added in slice order
// (deterministic); red holds each thread's 4 x 4 block.
template <typename T>
__device__ __forceinline__ void stash_acc(T* red, const T (&acc)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) red[threadIdx.x * 16 + u * 4 + w] = acc[u][w];
  __syncthreads();
}
template <typename T>
__device__ __forceinline__ void publish(const T* red, T* pub, int nbb, int nblk, int slices, int na,
                                        int nb) {
  for (int e = threadIdx.x; e < na * nb; e += kThreads) {
    const int a = e / nb, b = e % nb;
    const int blk = (a / 4) * nbb + b / 4, q = (a % 4) * 4 + b % 4;
    T s = 0;
    for (int sl = 0; sl < slices; ++sl) s += red[(sl * nblk + blk) * 16 + q];
    pub[e] = s;
  }
}

// sum[e] = sum over the cluster's ranks, in rank order, of their pub[e].
template <typename T>
__device__ __forceinline__ void cluster_sum(T* pub, T* sum, cg::cluster_group& cluster, int ne,
                                            int cs) {
  cluster.sync();   // every rank has published
  for (int e = threadIdx.x; e < ne; e += kThreads) {
    T v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = q < cs ? cluster.map_shared_rank(pub, q)[e] : T(0);
    T s = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) s += v[q];
    sum[e] = s;
  }
  __syncthreads();
}

// Warp 0: Cholesky A = R^T R in place on the n x n Gram in A (upper
// triangle read, R written over it), lane j holding column j in registers;
// the pivot row is passed between lanes by shuffles.  A pivot below droptol
// times the largest diagonal entry marks its column as dependent on the
// earlier ones: its row of R and its entry of rdiag (= 1 / R[k][k]) are
// zero, so the matching column of Q comes out zero and drops out of both the
// head and the tail projection.  In fp32, 1 / R[k][k] is the hardware
// reciprocal square root (within 2 ulp); the second CholeskyQR pass absorbs
// that.  The former loop over shared memory took 3.6 us per factorisation
// (a chain of shared-memory round trips per column update, per timestamps);
// not inlined, so that one warm-up run fetches its code before the first
// real use (see stage_tile).
template <typename T>
__device__ __noinline__ void cholesky(T (*A)[kMaxR + 1], int n, T* rdiag, T droptol) {
  const int j = threadIdx.x & 31;
  T col[kMaxR];
  T diag = T(0);
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    col[i] = (j < n && i <= j) ? A[i][j] : T(0);
    if (i == j) diag = col[i];
  }
  T dmax = diag;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dmax = fmax(dmax, __shfl_xor_sync(0xffffffffu, dmax, off));
  const T tol = droptol * dmax;
#pragma unroll
  for (int k = 0; k < kMaxR; ++k) {
    if (k >= n) break;
    const T piv = __shfl_sync(0xffffffffu, col[k], k);
    const bool keep = piv > tol && dmax > T(0);
    const T inv = keep ? rsqrt_t(piv) : T(0);
    col[k] = j == k ? piv * inv : (j > k ? col[k] * inv : col[k]);
    if (j == k) rdiag[k] = inv;
    // A[i2][j] -= R[k][i2] R[k][j] for k < i2 <= j
#pragma unroll
    for (int i2 = k + 1; i2 < kMaxR; ++i2) {
      const T rki2 = __shfl_sync(0xffffffffu, col[k], i2);
      if (j >= i2) col[i2] = fma(-rki2, col[k], col[i2]);
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxR; ++i)
    if (j < n && i <= j) A[i][j] = col[i];
  __syncwarp();
}

// In place on the staged rows [0, nrows): x[c, :] <- x[c, :] M over the first
// r columns.  One thread per row.
__device__ __forceinline__ void apply_matrix(Smem& sm, const float (*M)[kMaxR], int r, int nrows) {
  for (int c = threadIdx.x; c < nrows; c += kThreads) {
    float q[kMaxR];
#pragma unroll
    for (int b = 0; b < kMaxR; ++b) q[b] = 0.f;
    for (int a = 0; a < r; ++a) {
      const float xa = sm.xs[a][c];
#pragma unroll
      for (int b4 = 0; b4 < kMaxR; b4 += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(&M[a][b4]);
        q[b4] = fmaf(xa, m4.x, q[b4]);
        q[b4 + 1] = fmaf(xa, m4.y, q[b4 + 1]);
        q[b4 + 2] = fmaf(xa, m4.z, q[b4 + 2]);
        q[b4 + 3] = fmaf(xa, m4.w, q[b4 + 3]);
      }
    }
#pragma unroll
    for (int b = 0; b < kMaxR; ++b)
      if (b < r) sm.xs[b][c] = q[b];
  }
}

// In place on the staged rows [0, nrows), after Q: g columns <- W = G' - Q
// (Q^T G').  One thread per row, its Q row in registers.
__device__ __forceinline__ void tail_rows(Smem& sm, int r, int m, int nrows) {
  for (int c = threadIdx.x; c < nrows; c += kThreads) {
    float q[kMaxR];
#pragma unroll
    for (int a = 0; a < kMaxR; ++a) q[a] = a < r ? sm.xs[a][c] : 0.f;
    for (int l = 0; l < m; ++l) {
      const float* cm = sm.CmT[l];
      float s0 = sm.xs[r + l][c], s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int a = 0; a < kMaxR; a += 4) {
        const float4 v = *reinterpret_cast<const float4*>(cm + a);
        s0 = fmaf(-q[a], v.x, s0);
        s1 = fmaf(-q[a + 1], v.y, s1);
        s2 = fmaf(-q[a + 2], v.z, s2);
        s3 = fmaf(-q[a + 3], v.w, s3);
      }
      sm.xs[r + l][c] = (s0 + s1) + (s2 + s3);
    }
  }
}

// Output rows [0, nrows) of the tile at global row `base`: [Q | W | 0] from
// the staged columns.  Items of 8 consecutive rows x one column; 16-byte
// stores when the row range allows them.
__device__ __forceinline__ void write_rows(const Smem& sm, const HppQrParams& p, int i, int base,
                                           int nrows) {
  const int nc = p.r + p.m;
  const int groups = (nrows + 7) / 8;
  const bool vec = (p.p % 8) == 0;   // then base and every column start are 16-byte aligned (bf16)
  for (int e = threadIdx.x; e < kMaxNP * groups; e += kThreads) {
    const int j = e / groups, c0 = (e % groups) * 8;
    float v[8];
    if (j < nc) {
      const float4 x0 = *reinterpret_cast<const float4*>(&sm.xs[j][c0]);
      const float4 x1 = *reinterpret_cast<const float4*>(&sm.xs[j][c0 + 4]);
      v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
      v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = 0.f;
    }
    const size_t o = ((size_t)i * kMaxNP + j) * p.p + base + c0;
    if (p.out_f32) {
      for (int u = 0; u < 8 && c0 + u < nrows; ++u) p.out_f32[o + u] = v[u];
    } else if (vec && c0 + 8 <= nrows) {
      __align__(16) __nv_bfloat16 hi[8], lo[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) split_hilo(v[u], hi[u], lo[u]);
      *reinterpret_cast<uint4*>(p.out_hi + o) = *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(p.out_lo + o) = *reinterpret_cast<const uint4*>(lo);
    } else {
      for (int u = 0; u < 8 && c0 + u < nrows; ++u) {
        __nv_bfloat16 hi, lo;
        split_hilo(v[u], hi, lo);
        p.out_hi[o + u] = hi;
        p.out_lo[o + u] = lo;
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void zero_acc(T (&acc)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) acc[u][w] = T(0);
}

// kF64: the first pass's Gram, Cholesky factor and inverse in fp64 (fp32
// inputs); its shared memory follows Smem.
template <bool kF64>
__global__ void __launch_bounds__(kThreads, 1) hpp_qr_kernel(const __grid_constant__ HppQrParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  Smem64& s64 = *reinterpret_cast<Smem64*>(smem_raw + ((sizeof(Smem) + 15) & ~size_t(15)));
  cg::cluster_group cluster = cg::this_cluster();
  pdl_trigger();
  pdl_wait();
  const int cs = p.cs;
  const int i = (int)blockIdx.x / cs;               // one cluster per sample
  const int rank = (int)cluster.block_rank();
  const int r = p.r, m = p.m;
  const int per = (((p.p + cs - 1) / cs) + 7) / 8 * 8;
  const int row0 = min(p.p, rank * per);
  const int row_end = min(p.p, row0 + per);
  const int nt = max(1, (row_end - row0 + kTileRows - 1) / kTileRows);
  const bool resident = nt == 1;

  // pass 0: Gram V^T V -> R1.  pass 1: Q1 = V R1^-1, one reduction for both
  // Q1^T Q1 (close to the identity) -> R2 and K = Q1^T G'; then Q = Q1 R2^-1
  // and Q^T G' = R2^-T K.  pass 2: outputs [Q | W | 0].  A resident tile is
  // staged once and transformed in place; otherwise every pass re-stages
  // each tile and re-applies the factors it needs.
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int nb = pass == 0 ? r : r + m;
    const Blocking bk(r, nb);
    const bool f64 = kF64 && pass == 0;
    float acc[4][4];
    double acc64[4][4];
    zero_acc(acc);
    if (kF64) zero_acc(acc64);
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      const int base = row0 + t * kTileRows;
      const int nv = max(0, min(kTileRows, row_end - base));
      if (pass == 0 || !resident) stage_tile(sm, p, i, base, nv, pass == 0 && t == 0);
      const int first = (pass == 0 || (resident && pass == 2)) ? 2 : 1;
      const int last = pass == 2 ? 2 : pass;   // factors applied: M1 (1), M2 (2)
#pragma unroll 1
      for (int f = first; f <= last; ++f) {
        apply_matrix(sm, f == 1 ? sm.M1 : sm.M2, r, nv);
        __syncthreads();
      }
      if (f64) {
        accumulate(sm, bk, nv, acc64);
      } else if (pass < 2) {
        accumulate(sm, bk, nv, acc);
      } else {
        tail_rows(sm, r, m, nv);
        __syncthreads();
        write_rows(sm, p, i, base, nv);
      }
      if (!resident) __syncthreads();
    }
    if (pass == 2) break;
    if (f64) {
      stash_acc(s64.red, acc64);
      publish(s64.red, s64.pub, bk.nbb, bk.nblk, bk.slices, r, nb);
      cluster_sum(s64.pub, s64.sum, cluster, r * nb, cs);
      for (int e = threadIdx.x; e < r * r; e += kThreads) s64.R[e / r][e % r] = s64.sum[e];
      __syncthreads();
      if (threadIdx.x < 32) cholesky(s64.R, r, s64.rd, kDropTol64);
      __syncthreads();
      if (threadIdx.x < 32) invert_factor(s64.R, s64.rd, r, sm.M1);
      __syncthreads();
      continue;
    }
    stash_acc(sm.red, acc);
    publish(sm.red, sm.pub[pass], bk.nbb, bk.nblk, bk.slices, r, nb);
    cluster_sum(sm.pub[pass], sm.sum, cluster, r * nb, cs);
    float (*R)[kMaxR + 1] = pass == 0 ? sm.R1 : sm.R2;
    for (int e = threadIdx.x; e < r * nb; e += kThreads) {
      const int a = e / nb, b = e % nb;
      if (b < r) R[a][b] = sm.sum[e];
      else sm.K[a][b - r] = sm.sum[e];
    }
    __syncthreads();
    float* rd = pass == 0 ? sm.rd1 : sm.rd2;
    if (threadIdx.x < 32) cholesky(R, r, rd, kDropTol);
    __syncthreads();
    if (threadIdx.x < 32) invert_factor<float>(R, rd, r, pass == 0 ? sm.M1 : sm.M2);
    __syncthreads();
    if (pass == 1) {
      // Cm = R2^-T K = M2^T K, stored transposed; one entry per thread
      for (int e = threadIdx.x; e < kMaxM * kMaxR; e += kThreads) {
        const int l = e / kMaxR, b = e % kMaxR;
        float s2 = 0.f;
        if (l < m)
          for (int a = 0; a <= b && a < r; ++a) s2 = fmaf(sm.M2[a][b], sm.K[a][l], s2);
        sm.CmT[l][b] = s2;
      }
      __syncthreads();
    }
  }
  // the other ranks may still be reading this CTA's partials
  cluster.sync();
}

// Largest cluster this kernel can be launched with on the current device:
// 16 CTAs (a non-portable size) where the device has room for one, else 8.
// Cached per device and shared-memory size (atomics: calls may come from
// several host threads).
template <bool kF64>
int cluster_cap(size_t smem) {
  static std::atomic<int> cap[16];
  static std::atomic<size_t> cap_smem[16];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) dev = 0;
  const int cached = cap[dev].load(std::memory_order_acquire);
  if (cached && cap_smem[dev].load(std::memory_order_relaxed) == smem) return cached;
  int c = 8;
  if (cudaFuncSetAttribute(hpp_qr_kernel<kF64>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 16;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, hpp_qr_kernel<kF64>, &cfg) == cudaSuccess && n > 0)
      c = 16;
  }
  (void)cudaGetLastError();
  cap_smem[dev].store(smem, std::memory_order_relaxed);
  cap[dev].store(c, std::memory_order_release);
  return c;
}

template <bool kF64>
cudaError_t launch_qr(const HppQrParams& p_in, cudaStream_t s) {
  const size_t smem = kF64 ? ((sizeof(Smem) + 15) & ~size_t(15)) + sizeof(Smem64) : sizeof(Smem);
  cudaError_t e = cudaFuncSetAttribute(hpp_qr_kernel<kF64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  HppQrParams p = p_in;
  p.cs = std::min(cluster_cap<kF64>(smem), std::max(1, (p.p + kRowsTarget - 1) / kRowsTarget));
  return launch_pdl(hpp_qr_kernel<kF64>, dim3(p.B * p.cs), dim3(kThreads), smem, s, p.cs, p);
}

}  // namespace

cudaError_t launch_hpp_qr(const HppQrParams& p_in, cudaStream_t s) {
  if (p_in.r < 1 || p_in.r > kMaxR || p_in.m > kMaxM || p_in.r + p_in.m > kMaxNP)
    return cudaErrorInvalidValue;
  return p_in.gram_f64 ? launch_qr<true>(p_in, s) : launch_qr<false>(p_in, s);
}

}  // namespace dpclip
