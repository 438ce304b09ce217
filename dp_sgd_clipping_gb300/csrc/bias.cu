// Bias of the linear layer ("Algorithmic flow" steps 3-5 of the randomized-
// clipping summary applied to every parameter; "DP-SGD algorithm" step 3
// clips the whole per-sample gradient).  For y_t = x_t W + b the per-sample
// bias gradient is b_i = sum_t G_i[t, :]: a column sum over the sample's
// tokens, which reads G once (HBM-bound, no tensor-core work).
//
//   bias_partial: CTA (column block of 256, token chunk, sample) -> the
//     chunk's column sums; warp w takes rows w, w + 8, ... of the chunk, lane
//     l eight consecutive columns (one 16-byte load of bf16 per row), and the
//     eight warps are added in warp order.
//   bias_finalize: CTA (column block, sample) adds the chunks in chunk order
//     (b_i) and the squares of its columns; bias_sq: one warp per sample adds
//     the column blocks in order, sqnorms[i] (+)= ||b_i||^2.
//   bias_clip: grad_b[c] = sum_i s_i b_i[c] + sigma C z_c, z from Philox
//     stream 4 at element c, samples added in index order.
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kBiasCols = 256;      // columns per CTA: 32 lanes x 8
constexpr int kBiasThreads = 256;   // 8 warps
constexpr int kBiasRowsUnroll = 8;  // rows in flight per warp

__device__ __forceinline__ void add8_bf16(const uint4 u, float (&acc)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    acc[2 * q] += f.x;
    acc[2 * q + 1] += f.y;
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kBiasThreads) bias_partial_kernel(const void* G, int T, int p,
                                                                    int chunk, float* part) {
  __shared__ float red[kBiasThreads / 32][kBiasCols];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cb = blockIdx.x, tc = blockIdx.y, i = blockIdx.z;
  const int c0 = cb * kBiasCols + lane * 8;
  const int t0 = tc * chunk, t1 = min(T, t0 + chunk);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  if (kBf16) {
    // p % 8 == 0 on this path: a lane's 8 columns are all in or all out
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(G) + (size_t)i * T * p;
    if (c0 < p) {
      int t = t0 + warp;
      for (; t + 8 * (kBiasRowsUnroll - 1) < t1; t += 8 * kBiasRowsUnroll) {
        uint4 u[kBiasRowsUnroll];
#pragma unroll
        for (int r = 0; r < kBiasRowsUnroll; ++r)
          u[r] = __ldcs(reinterpret_cast<const uint4*>(g + (size_t)(t + 8 * r) * p + c0));
#pragma unroll
        for (int r = 0; r < kBiasRowsUnroll; ++r) add8_bf16(u[r], acc);
      }
      for (; t < t1; t += 8)
        add8_bf16(__ldcs(reinterpret_cast<const uint4*>(g + (size_t)t * p + c0)), acc);
    }
  } else {
    const float* g = static_cast<const float*>(G) + (size_t)i * T * p;
    for (int t = t0 + warp; t < t1; t += 8) {
      const float* row = g + (size_t)t * p;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + q < p) acc[q] += row[c0 + q];
    }
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) red[warp][lane * 8 + q] = acc[q];
  __syncthreads();
  // column c of the block: the eight warps in order
  const int c = threadIdx.x;   // kBiasThreads == kBiasCols
  const int col = cb * kBiasCols + c;
  if (col < p) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kBiasThreads / 32; ++w) s += red[w][c];
    part[((size_t)i * gridDim.y + tc) * p + col] = s;
  }
}

__global__ void __launch_bounds__(kBiasCols) bias_finalize_kernel(const float* part, int nchunks,
                                                                 int p, float* bias,
                                                                 float* part2) {
  __shared__ float red[kBiasCols / 32];
  pdl_trigger();
  pdl_wait();
  const int cb = blockIdx.x, i = blockIdx.y;
  const int c = cb * kBiasCols + threadIdx.x;
  float b = 0.f;
  if (c < p) {
    for (int k = 0; k < nchunks; ++k) b += part[((size_t)i * nchunks + k) * p + c];
    if (bias) bias[(size_t)i * p + c] = b;
  }
  float ss = warp_sum(b * b);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kBiasCols / 32; ++w) s += red[w];
    part2[(size_t)i * gridDim.x + cb] = s;
  }
}

__global__ void bias_sq_kernel(const float* part2, int ncb, int B, float* sq, int accumulate) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= B) return;
  float s = 0.f;
  for (int c0 = 0; c0 < ncb; c0 += 32) s += c0 + lane < ncb ? part2[(size_t)i * ncb + c0 + lane] : 0.f;
  s = warp_sum(s);
  if (lane == 0) sq[i] = accumulate ? sq[i] + s : s;
}

__global__ void bias_clip_kernel(const float* bias, int B, int p, const float* sq, float C,
                                 float nscale, uint64_t seed, uint64_t offset, float* grad_b,
                                 float* param, float upd_scale, const FiberDev fiber,
                                 int use_fiber) {
  extern __shared__ float s_sh[];
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const float q = sq[i];
    s_sh[i] = q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
  }
  __syncthreads();
  const int nb = (p + 3) / 4;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < nb; b += gridDim.x * blockDim.x) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < B; ++i) {
      const float si = s_sh[i];
#pragma unroll
      for (int l = 0; l < 4; ++l)
        if (4 * b + l < p) acc[l] = fmaf(si, bias[(size_t)i * p + 4 * b + l], acc[l]);
    }
    if (nscale != 0.f) {
      float z[4];
      philox_normal4_fast(seed, 4u, offset, (uint32_t)b, z);
#pragma unroll
      for (int l = 0; l < 4; ++l) acc[l] = fmaf(nscale, z[l], acc[l]);
    }
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      if (4 * b + l < p) {
        if (grad_b) grad_b[4 * b + l] = acc[l];
        if (param) param[4 * b + l] = fmaf(-upd_scale, acc[l], param[4 * b + l]);
        if (use_fiber) fiber_update1(fiber, 4 * (size_t)b + l, acc[l]);
      }
    }
  }
}

}  // namespace

int bias_chunk_rows(int T) { return T <= 512 ? T : 512; }
int bias_nchunks(int T) { return (T + bias_chunk_rows(T) - 1) / bias_chunk_rows(T); }
size_t bias_part_floats(int B, int T, int p) {
  return (size_t)B * bias_nchunks(T) * p + (size_t)B * ((p + kBiasCols - 1) / kBiasCols);
}

cudaError_t launch_bias_grads(const void* G, bool bf16, int B, int T, int p, float* part,
                              float* bias, float* sq, int accumulate, cudaStream_t s) {
  const int chunk = bias_chunk_rows(T), nchunks = bias_nchunks(T);
  const int ncb = (p + kBiasCols - 1) / kBiasCols;
  float* part2 = part + (size_t)B * nchunks * p;
  const dim3 grid(ncb, nchunks, B);
  cudaError_t e =
      bf16 ? launch_pdl(bias_partial_kernel<true>, grid, dim3(kBiasThreads), 0, s, 0, G, T, p, chunk,
                        part)
           : launch_pdl(bias_partial_kernel<false>, grid, dim3(kBiasThreads), 0, s, 0, G, T, p,
                        chunk, part);
  if (e != cudaSuccess) return e;
  e = launch_pdl(bias_finalize_kernel, dim3(ncb, B), dim3(kBiasCols), 0, s, 0, (const float*)part,
                 nchunks, p, bias, part2);
  if (e != cudaSuccess || !sq) return e;
  return launch_pdl(bias_sq_kernel, dim3((B + 7) / 8), dim3(256), 0, s, 0, (const float*)part2, ncb,
                    B, sq, accumulate);
}

cudaError_t launch_bias_clip(const float* bias, int B, int p, const float* sq, float C, float nscale,
                             uint64_t seed, uint64_t offset, float* grad_b, float* param,
                             float upd_scale, const FiberDev* fiber, cudaStream_t s) {
  const FiberDev fz = fiber ? *fiber : FiberDev{};
  const int nb = (p + 3) / 4;
  const int threads = 256;
  const int grid = std::max(1, std::min((nb + threads - 1) / threads, 152 * 4));
  return launch_pdl(bias_clip_kernel, dim3(grid), dim3(threads), (size_t)B * sizeof(float), s, 0,
                    bias, B, p, sq, C, nscale, seed, offset, grad_b, param, upd_scale, fz,
                    fiber ? 1 : 0);
}

}  // namespace dpclip
