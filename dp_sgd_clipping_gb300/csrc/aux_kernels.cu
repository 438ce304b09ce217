// Small kernels of the clipping path: Philox probe fill, clip scales,
// deterministic reduction of per-tile norm partials, gradient noise for the
// fp32 path and the bounded-wait self-test.
#include <algorithm>

#include "common.cuh"

namespace dpclip {
namespace {

// out (rows x cols, row-major) = probes of one Philox stream for the first
// rows_valid rows (element e = j * cols + c uses Philox block e / 4, lane
// e % 4), zeros below.  kind 0: standard normals (Box-Muller); kind 1:
// Rademacher values, +1 / -1 by the top bit of the lane's word.  One thread
// per Philox block of four elements; one launch fills up to two such
// matrices (jobs), the blocks of the second following those of the first.
struct FillJob {
  void* out;
  int64_t rows, cols, rows_valid;
  uint32_t stream_id;
};
struct FillJobs {
  FillJob job[2];
  int njobs;
};

template <bool kBf16>
__device__ __forceinline__ void fill_block(const FillJob& j, int64_t b, uint64_t seed,
                                           uint64_t offset, int kind) {
  const int64_t nvalid = j.rows_valid * j.cols, ntotal = j.rows * j.cols;
  float z[4] = {0.f, 0.f, 0.f, 0.f};
  if (4 * b < nvalid) {
    if (kind == 1) {
      const U4 x = philox4x32_10(U4{(uint32_t)b, j.stream_id, (uint32_t)offset,
                                    (uint32_t)(offset >> 32)},
                                 (uint32_t)seed, (uint32_t)(seed >> 32));
      z[0] = (x.x >> 31) ? -1.f : 1.f;
      z[1] = (x.y >> 31) ? -1.f : 1.f;
      z[2] = (x.z >> 31) ? -1.f : 1.f;
      z[3] = (x.w >> 31) ? -1.f : 1.f;
    } else {
      philox_normal4(seed, j.stream_id, offset, (uint32_t)b, z);
    }
  }
#pragma unroll
  for (int l = 0; l < 4; ++l) {
    const int64_t e = 4 * b + l;
    if (e >= ntotal) break;
    const float v = e < nvalid ? z[l] : 0.f;
    if (kBf16)
      static_cast<__nv_bfloat16*>(j.out)[e] = __float2bfloat16_rn(v);
    else
      static_cast<float*>(j.out)[e] = v;
  }
}

template <bool kBf16>
__global__ void philox_fill_kernel(const FillJobs jobs, uint64_t seed, uint64_t offset,
                                   uint32_t* zero, int zero_words, int kind) {
  // the first kernel of a Hutch / Hutch++ call: its dependents may read the
  // call's inputs before their own wait, so they start only once everything
  // before the call has completed
  pdl_wait();
  pdl_trigger();
  if (zero)
    for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < zero_words; w += gridDim.x * blockDim.x)
      zero[w] = 0u;
  const int64_t nblk0 = (jobs.job[0].rows * jobs.job[0].cols + 3) / 4;
  const int64_t nblk1 = jobs.njobs > 1 ? (jobs.job[1].rows * jobs.job[1].cols + 3) / 4 : 0;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblk0 + nblk1;
       b += (int64_t)gridDim.x * blockDim.x) {
    if (b < nblk0)
      fill_block<kBf16>(jobs.job[0], b, seed, offset, kind);
    else
      fill_block<kBf16>(jobs.job[1], b - nblk0, seed, offset, kind);
  }
}

// Zeroes a call's control words (error word, tickets) once the previous
// kernel of the stream has completed; a programmatic launch, so the call's
// next kernel sets itself up meanwhile.
__global__ void clear_words_kernel(uint32_t* w, int n) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) w[i] = 0u;
}

__global__ void clip_scales_kernel(const float* sq, int B, float C, float* scales, uint8_t* clipped) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B; i += gridDim.x * blockDim.x) {
    const float q = sq[i];
    if (scales) scales[i] = q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
    if (clipped) clipped[i] = (uint8_t)(sqrtf(fmaxf(q, 0.f)) > C);
  }
}

// sq[i] = scale * sum over units u and slots w of part[(u*su + i*si)*nw + w];
// one block per sample, fixed summation tree.
__global__ void finalize_norms_kernel(const float* part, int nunits, long long su, long long si,
                                      int nw, float scale, float* sq, int accumulate) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x;
  const long long n = (long long)nunits * nw;
  float acc = 0.f;
  for (long long e = threadIdx.x; e < n; e += blockDim.x) {
    const long long u = e / nw, w = e % nw;
    acc += part[(u * su + (long long)i * si) * nw + w];
  }
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    sq[i] = accumulate ? sq[i] + scale * s : scale * s;
  }
}

// Stored per-sample gradients -> clipped noisy sum ("DP-SGD algorithm" steps
// 3-4 of the DP-SGD glossary): one thread per Philox block of four elements,
// the samples added in index order.
__global__ void stored_grad_kernel(const float* __restrict__ M, int B, long long n,
                                   long long stride, const float* sq, float C, float nscale,
                                   uint64_t seed, uint64_t offset, float* grad, float* scales,
                                   uint8_t* clipped, float* param, float upd_scale,
                                   const FiberDev fiber, int use_fiber) {
  extern __shared__ float s_sh[];
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const float q = sq[i];
    const float si = q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
    s_sh[i] = si;
    if (blockIdx.x == 0) {
      if (scales) scales[i] = si;
      if (clipped) clipped[i] = (uint8_t)(sqrtf(fmaxf(q, 0.f)) > C);
    }
  }
  __syncthreads();
  const long long nb = (n + 3) / 4, s4 = stride / 4;
  const float4* M4 = reinterpret_cast<const float4*>(M);
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb;
       b += (long long)gridDim.x * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int i = 0;
    for (; i + 4 <= B; i += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(M4 + (size_t)(i + u) * s4 + b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float si = s_sh[i + u];
        acc.x = fmaf(si, v[u].x, acc.x);
        acc.y = fmaf(si, v[u].y, acc.y);
        acc.z = fmaf(si, v[u].z, acc.z);
        acc.w = fmaf(si, v[u].w, acc.w);
      }
    }
    for (; i < B; ++i) {
      const float4 v = __ldcs(M4 + (size_t)i * s4 + b);
      const float si = s_sh[i];
      acc.x = fmaf(si, v.x, acc.x);
      acc.y = fmaf(si, v.y, acc.y);
      acc.z = fmaf(si, v.z, acc.z);
      acc.w = fmaf(si, v.w, acc.w);
    }
    if (nscale != 0.f) {
      float z[4];
      philox_normal4_fast(seed, 3u, offset, (uint32_t)b, z);
      acc.x = fmaf(nscale, z[0], acc.x);
      acc.y = fmaf(nscale, z[1], acc.y);
      acc.z = fmaf(nscale, z[2], acc.z);
      acc.w = fmaf(nscale, z[3], acc.w);
    }
    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
    if (4 * b + 3 < n) {
      if (grad) reinterpret_cast<float4*>(grad)[b] = acc;
      if (param) {   // the fused parameter update: theta -= (lr / L) g
        float4 w = reinterpret_cast<const float4*>(param)[b];
        w.x = fmaf(-upd_scale, acc.x, w.x);
        w.y = fmaf(-upd_scale, acc.y, w.y);
        w.z = fmaf(-upd_scale, acc.z, w.z);
        w.w = fmaf(-upd_scale, acc.w, w.w);
        reinterpret_cast<float4*>(param)[b] = w;
      }
      if (use_fiber) fiber_update4(fiber, 4 * (size_t)b, acc);
    } else {   // ragged end: lanes past n hold padding and are not stored
      for (int l = 0; 4 * b + l < n; ++l) {
        if (grad) grad[4 * b + l] = a4[l];
        if (param) param[4 * b + l] = fmaf(-upd_scale, a4[l], param[4 * b + l]);
        if (use_fiber) fiber_update1(fiber, 4 * (size_t)b + l, a4[l]);
      }
    }
  }
}

// An empty lot (no samples): g = nscale z from Philox stream `stream_id`
// (element e), stored to grad and / or applied as param -= upd_scale g.
__global__ void noise_only_kernel(float* grad, float* param, long long n, float nscale,
                                  float upd_scale, uint64_t seed, uint32_t stream_id,
                                  uint64_t offset, const FiberDev fiber, int use_fiber) {
  pdl_trigger();
  pdl_wait();
  const long long nblk = (n + 3) / 4;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblk;
       b += (long long)gridDim.x * blockDim.x) {
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    if (nscale != 0.f) philox_normal4_fast(seed, stream_id, offset, (uint32_t)b, z);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const long long e = 4 * b + l;
      if (e < n) {
        const float g = nscale * z[l];
        if (grad) grad[e] = g;
        if (param) param[e] = fmaf(-upd_scale, g, param[e]);
        if (use_fiber) fiber_update1(fiber, (size_t)e, g);
      }
    }
  }
}

// The FIBER step over a gradient already formed.
__global__ void fiber_kernel(const float* grad, long long n, const FiberDev f) {
  pdl_trigger();
  pdl_wait();
  const long long nb = (n + 3) / 4;
  const bool vec = (reinterpret_cast<uintptr_t>(grad) | reinterpret_cast<uintptr_t>(f.param) |
                    reinterpret_cast<uintptr_t>(f.filt) | reinterpret_cast<uintptr_t>(f.resid) |
                    reinterpret_cast<uintptr_t>(f.m) | reinterpret_cast<uintptr_t>(f.v)) % 16 == 0;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb;
       b += (long long)gridDim.x * blockDim.x) {
    if (vec && 4 * b + 3 < n) {
      fiber_update4(f, 4 * (size_t)b, reinterpret_cast<const float4*>(grad)[b]);
    } else {
      for (long long e = 4 * b; e < n && e < 4 * b + 4; ++e) fiber_update1(f, (size_t)e, grad[e]);
    }
  }
}

// param[e] -= scale * grad[e] (the update of the fp32 gradient path).
__global__ void sgd_update_kernel(float* param, const float* grad, long long n, float scale) {
  pdl_trigger();
  pdl_wait();
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    param[e] = fmaf(-scale, grad[e], param[e]);
}

// part[i * nblk + b] = sum of squares of elements [b c, (b + 1) c) of sample i
// (at M + i * stride), c = ceil(n / nblk); fixed summation tree.
__global__ void stored_sqnorm_kernel(const float* __restrict__ M, long long n, long long stride,
                                     float* part) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.y, nblk = gridDim.x;
  const long long chunk = (n + nblk - 1) / nblk;
  const long long e0 = blockIdx.x * chunk, e1 = min(n, e0 + chunk);
  const float* m = M + (size_t)i * stride;
  float acc = 0.f;
  for (long long e = e0 + threadIdx.x; e < e1; e += blockDim.x) acc = fmaf(m[e], m[e], acc);
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    part[(size_t)i * nblk + blockIdx.x] = s;
  }
}

__global__ void noise_add_kernel(float* grad, long long n, float scale, uint64_t seed,
                                 uint64_t offset) {
  pdl_trigger();
  pdl_wait();
  const long long nblk = (n + 3) / 4;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblk;
       b += (long long)gridDim.x * blockDim.x) {
    float z[4];
    philox_normal4_fast(seed, 3u, offset, (uint32_t)b, z);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const long long e = 4 * b + l;
      if (e < n) grad[e] = fmaf(scale, z[l], grad[e]);
    }
  }
}

// Waits on a barrier that nothing completes; the bounded wait gives up after
// limit_ns, records DPCLIP_ERR_TIMEOUT and the kernel returns normally.
__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, err, limit_ns};
    mbar_wait(&bar, 0, wc);
  }
}

}  // namespace

namespace {
cudaError_t launch_fill_jobs(const FillJobs& jobs, bool bf16, uint64_t seed, uint64_t offset,
                             cudaStream_t s, uint32_t* zero, int zero_words, int kind) {
  int64_t nblk = 0;
  for (int j = 0; j < jobs.njobs; ++j) nblk += (jobs.job[j].rows * jobs.job[j].cols + 3) / 4;
  const int threads = 256;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((nblk + threads - 1) / threads, 152 * 16));
  if (bf16)
    return launch_pdl(philox_fill_kernel<true>, dim3(grid), dim3(threads), 0, s, 0, jobs, seed,
                      offset, zero, zero_words, kind);
  return launch_pdl(philox_fill_kernel<false>, dim3(grid), dim3(threads), 0, s, 0, jobs, seed,
                    offset, zero, zero_words, kind);
}
}  // namespace

cudaError_t launch_philox_fill(void* out, int64_t rows, int64_t cols, int64_t rows_valid, bool bf16,
                               uint64_t seed, uint32_t stream_id, uint64_t offset, cudaStream_t s,
                               uint32_t* zero, int zero_words, int kind) {
  FillJobs jobs{};
  jobs.job[0] = FillJob{out, rows, cols, rows_valid, stream_id};
  jobs.njobs = 1;
  return launch_fill_jobs(jobs, bf16, seed, offset, s, zero, zero_words, kind);
}

cudaError_t launch_philox_fill2(void* out0, int64_t rows0, int64_t valid0, uint32_t stream0,
                                void* out1, int64_t rows1, int64_t valid1, uint32_t stream1,
                                int64_t cols, bool bf16, uint64_t seed, uint64_t offset,
                                cudaStream_t s, uint32_t* zero, int zero_words, int kind) {
  FillJobs jobs{};
  jobs.job[0] = FillJob{out0, rows0, cols, valid0, stream0};
  jobs.job[1] = FillJob{out1, rows1, cols, valid1, stream1};
  jobs.njobs = 2;
  return launch_fill_jobs(jobs, bf16, seed, offset, s, zero, zero_words, kind);
}

cudaError_t launch_clear_words(uint32_t* w, int n, cudaStream_t s) {
  const int threads = 256;
  const int grid = std::max(1, std::min((n + threads - 1) / threads, 152));
  return launch_pdl(clear_words_kernel, dim3(grid), dim3(threads), 0, s, 0, w, n);
}

cudaError_t launch_clip_scales(const float* sq, int B, float C, float* scales, uint8_t* clipped,
                               cudaStream_t s) {
  const int threads = 256;
  const int grid = std::min((B + threads - 1) / threads, 1024);
  return launch_pdl(clip_scales_kernel, dim3(grid), dim3(threads), 0, s, 0, sq, B, C, scales,
                    clipped);
}

cudaError_t launch_finalize_norms(const float* part, int B, int nunits, long long su, long long si,
                                  int nw, float scale, float* sq, cudaStream_t s, int accumulate) {
  return launch_pdl(finalize_norms_kernel, dim3(B), dim3(256), 0, s, 0, part, nunits, su, si,
                    nw, scale, sq, accumulate);
}

cudaError_t launch_stored_grad(const float* M, int B, long long n, long long stride,
                               const float* sq, float C, float nscale, uint64_t seed,
                               uint64_t offset, float* grad, float* scales, uint8_t* clipped,
                               float* param, float upd_scale, const FiberDev* fiber,
                               cudaStream_t s) {
  const FiberDev fz = fiber ? *fiber : FiberDev{};
  const long long nb = (n + 3) / 4;
  const int threads = 256;
  const int grid = (int)std::max<long long>(1, std::min<long long>((nb + threads - 1) / threads,
                                                                   152 * 8));
  return launch_pdl(stored_grad_kernel, dim3(grid), dim3(threads), (size_t)B * sizeof(float), s,
                    0, M, B, n, stride, sq, C, nscale, seed, offset, grad, scales, clipped, param,
                    upd_scale, fz, fiber ? 1 : 0);
}

cudaError_t launch_noise_only(float* grad, float* param, long long n, float nscale,
                              float upd_scale, uint64_t seed, uint32_t stream_id, uint64_t offset,
                              const FiberDev* fiber, cudaStream_t s) {
  const FiberDev fz = fiber ? *fiber : FiberDev{};
  const long long nblk = (n + 3) / 4;
  const int threads = 256;
  const int grid = (int)std::max<long long>(1, std::min<long long>((nblk + threads - 1) / threads,
                                                                   152 * 8));
  return launch_pdl(noise_only_kernel, dim3(grid), dim3(threads), 0, s, 0, grad, param, n, nscale,
                    upd_scale, seed, stream_id, offset, fz, fiber ? 1 : 0);
}

cudaError_t launch_fiber(const float* grad, long long n, const FiberDev& f, cudaStream_t s) {
  const long long nb = (n + 3) / 4;
  const int threads = 256;
  const int grid = (int)std::max<long long>(1, std::min<long long>((nb + threads - 1) / threads,
                                                                   152 * 8));
  return launch_pdl(fiber_kernel, dim3(grid), dim3(threads), 0, s, 0, grad, n, f);
}

cudaError_t launch_sgd_update(float* param, const float* grad, long long n, float scale,
                              cudaStream_t s) {
  const int threads = 256;
  const int grid = (int)std::max<long long>(1, std::min<long long>((n + threads - 1) / threads,
                                                                   152 * 8));
  return launch_pdl(sgd_update_kernel, dim3(grid), dim3(threads), 0, s, 0, param, grad, n, scale);
}

cudaError_t launch_stored_sqnorm(const float* M, int B, long long n, long long stride, int nblk,
                                 float* part, cudaStream_t s) {
  return launch_pdl(stored_sqnorm_kernel, dim3(nblk, B), dim3(256), 0, s, 0, M, n, stride, part);
}

cudaError_t launch_noise_add(float* grad, long long n, float scale, uint64_t seed, uint64_t offset,
                             cudaStream_t s) {
  const long long nblk = (n + 3) / 4;
  const int threads = 256;
  const int grid = (int)std::min<long long>((nblk + threads - 1) / threads, 152 * 16);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(noise_add_kernel, dim3(grid), dim3(threads), 0, s, 0, grad, n, scale, seed,
                    offset);
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace dpclip
