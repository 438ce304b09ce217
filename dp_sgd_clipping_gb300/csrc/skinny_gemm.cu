// Skinny tensor-core GEMMs of the randomized norm estimators.
//
// Hutch ("Core mechanism", item 1 of the randomized-clipping summary) needs,
// per sample i, Y_i = G_i P (T x k) and Z_i = A_i^T Y_i (d x k), then
// (1/k) ||Z_i||_F^2.  Both products stream one big operand (G or A) once and
// meet a skinny one (k <= 32 columns), so they are HBM-bound (32 flop/byte):
// the kernels below keep every SM's TMA queue deep and spend almost nothing
// on the tensor core.  Hutch++ (item 2) reuses the same two kernels for its
// three sweeps with other skinny operands.
//
//   tok_gemm:  out[i][j][t] = sum_f X[i][t][f] W[j][f]   (M = 128 tokens,
//              N = NP probe columns, K = features; X K-major via TMA)
//   feat_gemm: Z[i][f][j]   = sum_t X[i][t][f] Y[i][j][t] (M = 128 features,
//              N = NP, K = tokens; X MN-major via TMA, Y K-major)
//
// Skinny operands are bf16 hi + lo pairs (two MMAs into one fp32 TMEM
// accumulator), so a fp32 intermediate keeps ~16 significant bits.  A split
// of the K range over several CTAs is reduced deterministically inside a
// thread-block cluster: the splits of a tile are the CTAs of one cluster
// (along y).  CTA q of the cluster finishes the rows r with r % splits == q:
// every CTA stores its partial of those rows into CTA q's shared memory
// (posted stores), and after a cluster barrier CTA q adds them, in split
// order, from its own shared memory.  The former global round trip per
// partial (store, fence, ticket, reload by the last CTA) cost about 5 us of
// dependent latency at the end of every feature-side sweep, and pulling the
// partials over the cluster with remote loads about 3 us.
//
// Warp roles (128 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues
// tcgen05.mma, then all four warps drain TMEM (warp w owns TMEM lanes
// 32w..32w+31, i.e. tile rows 32w..32w+31).
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kStages = 4;   // 4 x 24 KB: two CTAs fit on one SM
constexpr uint32_t kXTileBytes = 128 * kBlockK * 2;   // 16 KB: 128 rows x 128 B

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint32_t tmem;
  int abort_flag;
  int is_last;
  int issued;
  int consumed;
  float red[4];
};

template <int NP>
__host__ __device__ constexpr uint32_t skinny_tile_bytes() {
  return (uint32_t)NP * 128u;   // NP rows x 64 bf16
}

template <int NP>
__host__ __device__ constexpr size_t skinny_smem_bytes() {
  return 1024 + (size_t)kStages * (kXTileBytes + 2 * skinny_tile_bytes<NP>()) + sizeof(SmemCtl);
}

// Drain after an abort: wait (bounded, not abortable) for the TMA loads that
// were issued but never consumed, and for the MMAs already issued, so that no
// async write lands in shared or tensor memory after the CTA has left.
__device__ void drain_after_abort(SmemCtl* ctl) {
  const uint64_t lim = 100000000ull;  // 100 ms per wait
  for (int it = ctl->consumed; it < ctl->issued; ++it) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&ctl->full[it % kStages], (uint32_t)(it / kStages) & 1u))
      if (globaltimer_ns() - t0 > lim) break;
  }
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(&ctl->done, 0))
    if (globaltimer_ns() - t0 > lim) break;
}

// Sum of one tile's K-split partials over the cluster that holds them (see
// the header).  z: this thread's row of this CTA's partial (row = thread);
// zs: this CTA's idle pipeline stages, which receive [splits][rows owned]
// rows of NP + 4 floats.  Returns true for the rows this CTA finishes
// (row % splits == rank), with their sums in z.  Every CTA of the cluster
// calls it (it holds two cluster barriers).
template <int NP>
__device__ __forceinline__ bool cluster_reduce_rows(float* zs, SmemCtl* ctl, float (&z)[32],
                                                    int row, int rank, int splits) {
  constexpr int ld = NP + 4;   // 16-byte rows, 4-bank stagger between rows
  const int rmax = (kTokTileM + splits - 1) / splits;
  __syncthreads();
  // no copy may still land in the stages that zs reuses
  if (ctl->abort_flag && threadIdx.x == 0) drain_after_abort(ctl);
  cluster_sync_all();   // every CTA's stages are idle: they may receive rows
  const int owner = row % splits, k = row / splits;
  const uint32_t dst = mapa_shared(smem_u32(zs + ((size_t)rank * rmax + k) * ld), (uint32_t)owner);
#pragma unroll
  for (int c = 0; c < NP / 4; ++c)
    st_dsmem_v4(dst + 16u * c, z[4 * c], z[4 * c + 1], z[4 * c + 2], z[4 * c + 3]);
  cluster_sync_all();   // every row has been delivered
  const bool mine = owner == rank;
  if (mine) {
#pragma unroll
    for (int j = 0; j < NP; ++j) z[j] = 0.f;
    for (int q = 0; q < splits; ++q) {
      const float* src = zs + ((size_t)q * rmax + k) * ld;
#pragma unroll
      for (int c = 0; c < NP / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(src + 4 * c);
        z[4 * c] += v.x;
        z[4 * c + 1] += v.y;
        z[4 * c + 2] += v.z;
        z[4 * c + 3] += v.w;
      }
    }
  }
  return mine;
}

// ---------------------------------------------------------------------------
// tok_gemm
// ---------------------------------------------------------------------------
template <int NP>
__global__ void __launch_bounds__(128, 1) tok_gemm_kernel(const __grid_constant__ TokGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr uint32_t kWBytes = skinny_tile_bytes<NP>();
  uint8_t* sX = smem;
  uint8_t* sWhi = sX + kStages * kXTileBytes;
  uint8_t* sWlo = sWhi + kStages * kWBytes;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(sWlo + kStages * kWBytes);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int i = tile / p.mtiles, mt = tile % p.mtiles;
  const int split = blockIdx.y;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(kb0 + p.kb_per_split, p.kblocks);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort_flag = 0;
    ctl->issued = 0;
    ctl->consumed = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_x);
    tma_prefetch_map(&p.map_whi);
    if (p.has_lo) tma_prefetch_map(&p.map_wlo);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // X (G or A) is an input of the call, and the call's first kernel starts
  // its dependents only once everything before the call has completed: the
  // first stages of X are requested before waiting for the previous kernel,
  // whose output (W) they do not need.
  const int nearly = min(kStages, nkb);
  const uint32_t bytes = kXTileBytes + kWBytes * (p.has_lo ? 2u : 1u);
  // each tile walks its K-blocks from its own starting point, so that the
  // CTAs in flight spread their row segments over the memory channels
  const int rot = nkb > 0 ? (int)(((unsigned)tile * 5u) % (unsigned)nkb) : 0;
  const uint64_t xpol = p.x_stream ? l2_evict_first_policy() : 0;
  auto load_x = [&](int st, int f) {
    if (p.x_stream)
      tma_load_3d_hint(sX + st * kXTileBytes, &p.map_x, &ctl->full[st], f, mt * kTokTileM, i, xpol);
    else
      tma_load_3d(sX + st * kXTileBytes, &p.map_x, &ctl->full[st], f, mt * kTokTileM, i);
  };
  if (warp == 0 && lane == 0) {
    for (int it = 0; it < nearly; ++it) {
      mbar_arrive_expect_tx(&ctl->full[it], bytes);
      load_x(it, (kb0 + (it + rot) % nkb) * kBlockK);
    }
  }
  pdl_wait();   // W may come from the previous kernel
  const uint32_t tmem = ctl->tmem;
  const WaitCtx wc{&ctl->abort_flag, p.err, kWaitLimitNs};

  if (warp == 0 && lane == 0) {
    const int wz = p.w_per_sample ? i : 0;
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kStages;
      const int f0 = (kb0 + (it + rot) % nkb) * kBlockK;
      if (it >= nearly) {
        if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&ctl->full[s], bytes);
        load_x(s, f0);
      }
      tma_load_3d(sWhi + s * kWBytes, &p.map_whi, &ctl->full[s], f0, 0, wz);
      if (p.has_lo) tma_load_3d(sWlo + s * kWBytes, &p.map_wlo, &ctl->full[s], f0, 0, wz);
      ctl->issued = it + 1;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, NP, false, false);
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kStages;
      if (!mbar_wait(&ctl->full[s], (it / kStages) & 1, wc)) break;
      ctl->consumed = it + 1;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sX + s * kXTileBytes);
      const uint32_t b0 = smem_u32(sWhi + s * kWBytes);
      const uint32_t c0 = smem_u32(sWlo + s * kWBytes);
#pragma unroll
      for (int kk = 0; kk < kBlockK / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, sdesc_sw128(b0 + kk * 32, 16, 1024), idesc, (it | kk) != 0);
        if (p.has_lo) umma_bf16(tmem, ad, sdesc_sw128(c0 + kk * 32, 16, 1024), idesc, 1);
      }
      umma_commit(&ctl->empty[s]);
    }
    umma_commit(&ctl->done);
  }
  __syncwarp();

  // ---- epilogue: all 4 warps, thread = one token row of the tile
  const int row = warp * 32 + lane;
  const int t = mt * kTokTileM + row;
  const size_t plane = (size_t)NP * p.Tp;
  // tcgen05.ld is warp-collective: decide per warp
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->done, 0, wc));
  float y[32];
  if (ok) {
    tc_fence_after();
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), y);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = 0.f;
  }
  bool mine = true;
  if (p.splits > 1)
    mine = cluster_reduce_rows<NP>(reinterpret_cast<float*>(sX), ctl, y, row, split, p.splits);
  if (mine) {
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      __nv_bfloat16 hi, lo;
      split_hilo(y[j], hi, lo);
      p.out_hi[(size_t)i * plane + (size_t)j * p.Tp + t] = hi;
      p.out_lo[(size_t)i * plane + (size_t)j * p.Tp + t] = lo;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (ctl->abort_flag && threadIdx.x == 0) drain_after_abort(ctl);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// ---------------------------------------------------------------------------
// feat_gemm
// ---------------------------------------------------------------------------
template <int NP, int MODE>
__global__ void __launch_bounds__(128, 1) feat_gemm_kernel(const __grid_constant__ FeatGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr uint32_t kYBytes = skinny_tile_bytes<NP>();
  constexpr uint32_t kHalf = 64 * 128;   // one 64-feature x 64-token box
  uint8_t* sX = smem;
  uint8_t* sYhi = sX + kStages * kXTileBytes;
  uint8_t* sYlo = sYhi + kStages * kYBytes;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(sYlo + kStages * kYBytes);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int i = tile / p.ftiles, ft = tile % p.ftiles;
  const int split = blockIdx.y;
  const int tb0 = split * p.tb_per_split;
  const int tb1 = min(tb0 + p.tb_per_split, p.tblocks);
  const int ntb = tb1 - tb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort_flag = 0;
    ctl->issued = 0;
    ctl->consumed = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_x);
    tma_prefetch_map(&p.map_yhi);
    tma_prefetch_map(&p.map_ylo);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // X (A or G) is an input of the call: its first stages are requested
  // before waiting for the previous kernel, whose output (Y) they do not
  // need (see tok_gemm_kernel).
  const int nearly = min(kStages, ntb);

  const uint32_t bytes = kXTileBytes + 2 * kYBytes;
  const int f0 = ft * kFeatTileM;
  const uint64_t xpol = p.x_stream ? l2_evict_first_policy() : 0;
  auto load_x = [&](int st, int t0) {
    if (p.x_stream && t0 < p.x_keep_t0) {
      tma_load_3d_hint(sX + st * kXTileBytes, &p.map_x, &ctl->full[st], f0, t0, i, xpol);
      tma_load_3d_hint(sX + st * kXTileBytes + kHalf, &p.map_x, &ctl->full[st], f0 + 64, t0, i,
                       xpol);
    } else {
      tma_load_3d(sX + st * kXTileBytes, &p.map_x, &ctl->full[st], f0, t0, i);
      tma_load_3d(sX + st * kXTileBytes + kHalf, &p.map_x, &ctl->full[st], f0 + 64, t0, i);
    }
  };
  if (warp == 0 && lane == 0) {
    for (int it = 0; it < nearly; ++it) {
      mbar_arrive_expect_tx(&ctl->full[it], bytes);
      load_x(it, (tb0 + it) * kBlockK);
    }
  }
  pdl_wait();   // Y may come from the previous kernel
  const uint32_t tmem = ctl->tmem;
  const WaitCtx wc{&ctl->abort_flag, p.err, kWaitLimitNs};

  if (warp == 0 && lane == 0) {
    for (int it = 0; it < ntb; ++it) {
      const int s = it % kStages;
      const int t0 = (tb0 + it) * kBlockK;
      if (it >= nearly) {
        if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&ctl->full[s], bytes);
        load_x(s, t0);
      }
      tma_load_3d(sYhi + s * kYBytes, &p.map_yhi, &ctl->full[s], t0, 0, i);
      tma_load_3d(sYlo + s * kYBytes, &p.map_ylo, &ctl->full[s], t0, 0, i);
      ctl->issued = it + 1;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, NP, true, false);
    for (int it = 0; it < ntb; ++it) {
      const int s = it % kStages;
      if (!mbar_wait(&ctl->full[s], (it / kStages) & 1, wc)) break;
      ctl->consumed = it + 1;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sX + s * kXTileBytes);
      const uint32_t b0 = smem_u32(sYhi + s * kYBytes);
      const uint32_t c0 = smem_u32(sYlo + s * kYBytes);
#pragma unroll
      for (int kk = 0; kk < kBlockK / 16; ++kk) {
        // MN-major A: 16 tokens = two 8-row groups of 1024 B; the two
        // 64-feature halves sit kHalf bytes apart.
        const uint64_t ad = sdesc_sw128(a0 + kk * 2048, kHalf, 1024);
        umma_bf16(tmem, ad, sdesc_sw128(b0 + kk * 32, 16, 1024), idesc, (it | kk) != 0);
        umma_bf16(tmem, ad, sdesc_sw128(c0 + kk * 32, 16, 1024), idesc, 1);
      }
      umma_commit(&ctl->empty[s]);
    }
    umma_commit(&ctl->done);
  }
  __syncwarp();

  // ---- epilogue: thread = one feature row of the tile
  const int row = warp * 32 + lane;
  const int f = ft * kFeatTileM + row;
  float z[32];
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->done, 0, wc));
  if (ok) {
    tc_fence_after();
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), z);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) z[j] = 0.f;
  }
  bool have_final = true;
  if (p.splits > 1)
    have_final = cluster_reduce_rows<NP>(reinterpret_cast<float*>(sX), ctl, z, row, split, p.splits);
  if (MODE == kFeatOutF32) {
    if (have_final && f < p.F) {
#pragma unroll
      for (int j = 0; j < NP; ++j) p.out_f32[((size_t)i * NP + j) * p.F + f] = z[j];
    }
  } else if (MODE == kFeatOutHiLo) {
    if (have_final && f < p.F) {
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        __nv_bfloat16 hi, lo;
        split_hilo(z[j], hi, lo);
        p.out_hi[((size_t)i * NP + j) * p.F + f] = hi;
        p.out_lo[((size_t)i * NP + j) * p.F + f] = lo;
      }
    }
  } else {
    // this CTA's share of the tile's weighted square sum: its finished rows
    float v = 0.f;
    if (have_final) {
#pragma unroll
      for (int j = 0; j < NP; ++j) v += p.w[j] * z[j] * z[j];
    }
    v = warp_sum(v);
    if (lane == 0) ctl->red[warp] = v;
    __syncthreads();
    const int nparts = p.ftiles * p.splits;
    uint32_t* cnt = p.counters + i;
    if (threadIdx.x == 0) {
      const float cta_sum = ((ctl->red[0] + ctl->red[1]) + ctl->red[2]) + ctl->red[3];
      p.qpart[(size_t)i * nparts + (size_t)ft * p.splits + split] = cta_sum;
      // release: this share is visible before the ticket is; acquire: the
      // last CTA's loads below (after the CTA barrier) see every share
      const uint32_t prev = atomic_add_acq_rel(cnt, 1u);
      ctl->is_last = (prev == (uint32_t)nparts - 1u);
    }
    __syncthreads();
    if (ctl->is_last && warp == 0) {
      // the last CTA of the sample adds the per-CTA sums: lane-parallel
      // loads, then a fixed shuffle tree (deterministic)
      float q = 0.f;
      for (int u0 = 0; u0 < nparts; u0 += 32) {
        const int u = u0 + lane;
        q += u < nparts ? __ldcg(p.qpart + (size_t)i * nparts + u) : 0.f;
      }
      q = warp_sum(q);
      if (lane == 0) {
        p.sq[i] = q;
        *cnt = 0u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (ctl->abort_flag && threadIdx.x == 0) drain_after_abort(ctl);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

size_t tok_gemm_smem(int NP) {
  return NP <= 16 ? skinny_smem_bytes<16>() : skinny_smem_bytes<32>();
}
size_t feat_gemm_smem(int NP) { return tok_gemm_smem(NP); }

// The K-splits of a tile form one cluster along y.
static dim3 split_cluster(int splits) {
  return splits > 1 ? dim3(1, (unsigned)splits, 1) : dim3(0, 0, 0);
}

cudaError_t launch_tok_gemm(const TokGemmParams& p, cudaStream_t s) {
  if (p.splits < 1 || p.splits > kMaxSplits) return cudaErrorInvalidValue;
  const dim3 grid(p.B * p.mtiles, p.splits);
  cudaError_t e;
  if (p.NP == 16) {
    const size_t sm = skinny_smem_bytes<16>();
    if ((e = set_smem(tok_gemm_kernel<16>, sm)) != cudaSuccess) return e;
    return launch_pdl_cluster(tok_gemm_kernel<16>, grid, dim3(128), sm, s,
                              split_cluster(p.splits), p);
  } else if (p.NP == 32) {
    const size_t sm = skinny_smem_bytes<32>();
    if ((e = set_smem(tok_gemm_kernel<32>, sm)) != cudaSuccess) return e;
    return launch_pdl_cluster(tok_gemm_kernel<32>, grid, dim3(128), sm, s,
                              split_cluster(p.splits), p);
  }
  return cudaErrorInvalidValue;
}

template <int NP, int MODE>
static cudaError_t launch_feat_t(const FeatGemmParams& p, cudaStream_t s) {
  const dim3 grid(p.B * p.ftiles, p.splits);
  const size_t sm = skinny_smem_bytes<NP>();
  cudaError_t e = set_smem(feat_gemm_kernel<NP, MODE>, sm);
  if (e != cudaSuccess) return e;
  return launch_pdl_cluster(feat_gemm_kernel<NP, MODE>, grid, dim3(128), sm, s,
                            split_cluster(p.splits), p);
}

cudaError_t launch_feat_gemm(const FeatGemmParams& p, int mode, cudaStream_t s) {
  if (p.splits < 1 || p.splits > kMaxSplits) return cudaErrorInvalidValue;
  if (p.NP == 16) {
    if (mode == kFeatOutF32) return launch_feat_t<16, kFeatOutF32>(p, s);
    if (mode == kFeatOutHiLo) return launch_feat_t<16, kFeatOutHiLo>(p, s);
    return launch_feat_t<16, kFeatSqNorm>(p, s);
  }
  if (p.NP == 32) {
    if (mode == kFeatOutF32) return launch_feat_t<32, kFeatOutF32>(p, s);
    if (mode == kFeatOutHiLo) return launch_feat_t<32, kFeatOutHiLo>(p, s);
    return launch_feat_t<32, kFeatSqNorm>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dpclip
