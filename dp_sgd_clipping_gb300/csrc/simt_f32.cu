// fp32 path: one tiled CUDA-core GEMM over a batch with strided operands and
// four epilogues, enough to express every product of the clipping path for
// float inputs (tf32 tensor cores would miss a 1e-5 relative tolerance).
//   acc_b(m, n) = sum_k X_b(m, k) * Y_b(k, n)
//   store:    out_b(m, n) = acc_b(m, n)
//   sqnorm:   part[b][block] = sum_{m,n} w(n) acc_b(m, n)^2
//   dot-with: part[b][block] = sum_{m,n} acc_b(m, n) * out_b(m, n)
//   grad:     out(m, n) = sum_b s_b acc_b(m, n),  s_b = min(1, C / sqrt(q_b))
// Tiles of 64 x 64 outputs, 256 threads, 4 x 4 outputs per thread, K in
// steps of 16 staged in shared memory.
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kTile = 64;
constexpr int kKStep = 16;

__device__ __forceinline__ float clip_scale(float q, float C) {
  return q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ SimtParams p, int mode) {
  __shared__ float xs[kKStep][kTile + 1];
  __shared__ float ys[kKStep][kTile + 1];
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  const int nblocks = gridDim.x * gridDim.y;
  const int blk = blockIdx.y * gridDim.x + blockIdx.x;

  const int b_begin = mode == kSimtGrad ? 0 : blockIdx.z;
  const int b_end = mode == kSimtGrad ? p.batch : blockIdx.z + 1;
  float tot[4][4] = {};
  for (int b = b_begin; b < b_end; ++b) {
    const float* X = p.X + (long long)b * p.xb;
    const float* Y = p.Y + (long long)b * p.yb;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < p.K; k0 += kKStep) {
      for (int e = threadIdx.x; e < kKStep * kTile; e += 256) {
        const int kk = e / kTile, mm = e % kTile;
        const int m = m0 + mm, k = k0 + kk;
        xs[kk][mm] = (m < p.M && k < p.K) ? X[(long long)m * p.xm + (long long)k * p.xk] : 0.f;
        const int n = n0 + mm;
        ys[kk][mm] = (n < p.N && k < p.K) ? Y[(long long)k * p.yk + (long long)n * p.yn] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kKStep; ++kk) {
        float xv[4], yv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) xv[r] = xs[kk][ty + 16 * r];
#pragma unroll
        for (int c = 0; c < 4; ++c) yv[c] = ys[kk][tx + 16 * c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(xv[r], yv[c], acc[r][c]);
      }
      __syncthreads();
    }
    if (mode == kSimtGrad) {
      const float s = clip_scale(p.sqnorms[b], p.C);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) tot[r][c] = fmaf(s, acc[r][c], tot[r][c]);
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) tot[r][c] = acc[r][c];
    }
  }

  const int b = b_begin;
  if (mode == kSimtStore || mode == kSimtGrad) {
    float* out = p.out + (mode == kSimtGrad ? 0 : (long long)b * p.ob);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = m0 + ty + 16 * r, n = n0 + tx + 16 * c;
        if (m < p.M && n < p.N) out[(long long)m * p.om + (long long)n * p.on] = tot[r][c];
      }
    return;
  }
  float v = 0.f;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int m = m0 + ty + 16 * r, n = n0 + tx + 16 * c;
      if (m < p.M && n < p.N) {
        if (mode == kSimtSqNorm) {
          const float w = p.w[n < 64 ? n : 63];
          v = fmaf(w * tot[r][c], tot[r][c], v);
        } else {
          v = fmaf(tot[r][c], p.out[(long long)b * p.ob + (long long)m * p.om + (long long)n * p.on], v);
        }
      }
    }
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w];
    p.part[(long long)b * nblocks + blk] = s;
  }
}

}  // namespace

int simt_nblocks(int M, int N) { return ((M + kTile - 1) / kTile) * ((N + kTile - 1) / kTile); }

cudaError_t launch_simt(const SimtParams& p, int mode, cudaStream_t s, int* nblocks_out) {
  const dim3 grid((p.N + kTile - 1) / kTile, (p.M + kTile - 1) / kTile,
                  mode == kSimtGrad ? 1 : p.batch);
  if (nblocks_out) *nblocks_out = (int)(grid.x * grid.y);
  return launch_pdl(simt_gemm_kernel, grid, dim3(256), 0, s, 0, p, mode);
}

}  // namespace dpclip
