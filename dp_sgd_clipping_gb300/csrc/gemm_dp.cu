// Per-sample weight-gradient tiles A_i^T G_i on the 5th-generation tensor core.
//
// Two epilogues share one persistent mainloop:
//   grad mode  ("DP-SGD algorithm" steps 3-4 of the DP-SGD glossary;
//               "Algorithmic flow" steps 4-5 of the randomized-clipping
//               summary): grad = sum_i s_i A_i^T G_i + sigma C Z with
//               s_i = min(1, C / sqrt(q_i)); the backward pass of the loss
//               rescaled by s_i is, for one linear layer, this scaled sum.
//   norm mode  (direct exact norm, the per-sample gradient materialisation of
//               "Problem definition", reduced on chip): partial sums of
//               (A_i^T G_i)^2, never storing the d x p tile.
//
// Work unit = (output tile of 128 d-rows x 256 p-columns, sample i).  In
// grad mode a CTA owns whole tiles (all B samples of a tile, which it folds
// into one running sum); in norm mode units are independent and are dealt
// out one by one (unit u = i * ntiles + tile, CTA c takes u = c, c + grid,
// ...), which evens out the last wave.  The K loop of a unit runs over that
// sample's T tokens in blocks of 64; both
// operands are MN-major (tokens are the slow axis of A and G), loaded by TMA
// with 128-byte swizzle.  The accumulator of a unit lives in TMEM (256
// columns); two accumulators alternate, so the epilogue of unit u overlaps
// the mainloop of unit u+1.  In grad mode the epilogue folds s_i * acc_i into
// a register-resident running sum (exact fp32 per-sample scaling) and, after
// the last sample of a tile, adds Philox noise and stores the tile.
//
// Roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2..9 = epilogue (warp w reads TMEM lanes 32*(w%4).., columns
// 128*((w-2)/4)..).
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kStages = 4;
constexpr uint32_t kBox = 64 * 128;              // 64 tokens x 128 B (64 bf16)
constexpr uint32_t kABytes = 2 * kBox;           // 128 d-columns
constexpr uint32_t kGBytes = 4 * kBox;           // 256 p-columns
constexpr int kThreads = 64 + 32 * kEpiWarps;    // 320

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem;
  int abort_flag;
  int issued;
  int consumed;
  int mma_units;     // units whose MMAs were committed to tfull
  int is_last;
  float red[kThreads / 32];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * (kABytes + kGBytes) + sizeof(Ctl);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float clip_scale(float q, float C) {
  return q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
}

__device__ __noinline__ void noise4(uint64_t seed, uint64_t offset, uint32_t blk, float4* z) {
  float v[4];
  philox_normal4(seed, 3u, offset, blk, v);
  *z = make_float4(v[0], v[1], v[2], v[3]);
}

// The k-th work unit of this CTA: (tile, sample).  Returns false past the end.
template <bool kGrad>
__device__ __forceinline__ bool unit_at(int k, int ntiles_total, int B, int& tile, int& i) {
  if (kGrad) {
    tile = (int)blockIdx.x + (k / B) * (int)gridDim.x;
    i = k % B;
    return tile < ntiles_total;
  }
  // sample-major: the CTAs running at the same time work on neighbouring
  // tiles of one sample and share its A and G slabs in L2
  const long long u = (long long)blockIdx.x + (long long)k * gridDim.x;
  i = (int)(u / ntiles_total);
  tile = (int)(u % ntiles_total);
  return u < (long long)ntiles_total * B;
}

template <bool kGrad>
__global__ void __launch_bounds__(kThreads, 1) gemm_dp_kernel(const __grid_constant__ GemmDpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sG = sA + kStages * kABytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(sG + kStages * kGBytes);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles_total = p.mtiles * p.ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 32 * kEpiWarps);
    }
    ctl->abort_flag = 0;
    ctl->issued = 0;
    ctl->consumed = 0;
    ctl->mma_units = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_a);
    tma_prefetch_map(&p.map_g);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();   // inputs (A, G, sqnorms) may come from the previous kernel
  if (kGrad && blockIdx.x == 0) {
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
      const float q = p.sqnorms[i];
      if (p.scales) p.scales[i] = clip_scale(q, p.C);
      if (p.clipped) p.clipped[i] = (uint8_t)(sqrtf(fmaxf(q, 0.f)) > p.C);
    }
  }
  const uint32_t tmem = ctl->tmem;
  const WaitCtx wc{&ctl->abort_flag, p.err, kWaitLimitNs};

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      int tile, i;
      for (int k = 0; unit_at<kGrad>(k, ntiles_total, p.B, tile, i); ++k) {
        const int d0 = (tile % p.mtiles) * kDpTileM;
        const int p0 = (tile / p.mtiles) * kDpTileN;
        bool run = true;
        for (int kb = 0; kb < p.tblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) {
            run = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->full[s], kABytes + kGBytes);
          const int t0 = kb * 64;
          uint8_t* a = sA + s * kABytes;
          uint8_t* g = sG + s * kGBytes;
          tma_load_3d(a, &p.map_a, &ctl->full[s], d0, t0, i);
          tma_load_3d(a + kBox, &p.map_a, &ctl->full[s], d0 + 64, t0, i);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tma_load_3d(g + q * kBox, &p.map_g, &ctl->full[s], p0 + 64 * q, t0, i);
          ctl->issued = it + 1;
        }
        if (!run) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, true, true);
      int it = 0;
      int tile, i;
      for (int u = 0; unit_at<kGrad>(u, ntiles_total, p.B, tile, i); ++u) {
        const int acc = u & 1;
        if (!mbar_wait(&ctl->tempty[acc], ((u >> 1) & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)acc * 256u;
        bool run = true;
        for (int kb = 0; kb < p.tblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->full[s], (it / kStages) & 1, wc)) {
            run = false;
            break;
          }
          ctl->consumed = it + 1;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t g0 = smem_u32(sG + s * kGBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_bf16(dt, sdesc_sw128(a0 + kk * 2048, kBox, 1024),
                      sdesc_sw128(g0 + kk * 2048, kBox, 1024), idesc, (kb | kk) != 0);
          }
          umma_commit(&ctl->empty[s]);
        }
        umma_commit(&ctl->tfull[acc]);
        ctl->mma_units = u + 1;
        if (!run) break;
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    float tot[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) tot[j] = 0.f;
    int tile, i;
    for (int u = 0; unit_at<kGrad>(u, ntiles_total, p.B, tile, i); ++u) {
      const int d0 = (tile % p.mtiles) * kDpTileM;
      const int p0 = (tile / p.mtiles) * kDpTileN;
      {
        const int acc = u & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->tfull[acc], (u >> 1) & 1, wc))) break;
        tc_fence_after();
        const uint32_t taddr =
            tmem + (uint32_t)acc * 256u + (uint32_t)half * 128u + ((uint32_t)(quad * 32) << 16);
        if (kGrad) {
          const float si = clip_scale(p.sqnorms[i], p.C);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float v[32];
            tmem_ld32(taddr + c4 * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              tot[c4 * 32 + j] = (i == 0) ? si * v[j] : fmaf(si, v[j], tot[c4 * 32 + j]);
          }
          tc_fence_before();
          mbar_arrive(&ctl->tempty[acc]);
        } else {
          float ss = 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float v[32];
            tmem_ld32(taddr + c4 * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
          }
          tc_fence_before();
          mbar_arrive(&ctl->tempty[acc]);
          ss = warp_sum(ss);
          if (lane == 0) p.part[((size_t)tile * p.B + i) * kEpiWarps + ew] = ss;
        }
        if (kGrad && i == p.B - 1) {
          const int r = d0 + quad * 32 + lane;
          const int cb = p0 + half * 128;
          if (r < p.d) {
            const float nscale = p.sigma * p.C;
            float* rowp = p.grad + (size_t)r * p.p;
#pragma unroll
            for (int jb = 0; jb < 32; ++jb) {
              const int c = cb + 4 * jb;
              if (c < p.p) {
                float4 o = make_float4(tot[4 * jb], tot[4 * jb + 1], tot[4 * jb + 2], tot[4 * jb + 3]);
                if (nscale != 0.f) {
                  float4 z;
                  noise4(p.seed, p.offset, (uint32_t)(((size_t)r * p.p + c) >> 2), &z);
                  o.x = fmaf(nscale, z.x, o.x);
                  o.y = fmaf(nscale, z.y, o.y);
                  o.z = fmaf(nscale, z.z, o.z);
                  o.w = fmaf(nscale, z.w, o.w);
                }
                *reinterpret_cast<float4*>(rowp + c) = o;
              }
            }
          }
        }
      }
    }
  }

  if (!kGrad)
    reduce_partials_last_cta(p.part, p.B, ntiles_total, p.B, 1, kEpiWarps, 1.f, p.sq, p.ticket,
                             ctl->red, &ctl->is_last);

  tc_fence_before();
  __syncthreads();
  if (ctl->abort_flag && threadIdx.x == 0) {
    // bounded drain of async work still in flight (loads, MMAs)
    const uint64_t lim = 100000000ull;
    for (int it = ctl->consumed; it < ctl->issued; ++it) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&ctl->full[it % kStages], (uint32_t)(it / kStages) & 1u))
        if (globaltimer_ns() - t0 > lim) break;
    }
    for (int a = 0; a < 2; ++a) {
      // the last committed use of accumulator a
      const int last_u = ctl->mma_units - 1 - ((ctl->mma_units - 1 - a) & 1);
      if (last_u < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&ctl->tfull[a], (uint32_t)(last_u >> 1) & 1u))
        if (globaltimer_ns() - t0 > lim) break;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t gemm_dp_smem() { return kSmemBytes; }

cudaError_t launch_gemm_dp(const GemmDpParams& p, bool grad_mode, int grid, cudaStream_t s) {
  cudaError_t e;
  if (grad_mode) {
    if ((e = cudaFuncSetAttribute(gemm_dp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess)
      return e;
    return launch_pdl(gemm_dp_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, s, false, p);
  }
  if ((e = cudaFuncSetAttribute(gemm_dp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes)) != cudaSuccess)
    return e;
  return launch_pdl(gemm_dp_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes, s, false, p);
}

}  // namespace dpclip
