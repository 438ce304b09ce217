// Exact per-sample squared norms in the ghost form
//   ||A_i^T G_i||_F^2 = sum_{t1,t2} (A_i A_i^T)[t1,t2] * (G_i G_i^T)[t1,t2],
// the Gram-Hadamard rewrite of the trace identity in "Core mechanism" of the
// randomized-clipping summary (the ghost-clipping baseline of its "Problem
// definition": O(T^2) per sample, no d x p tile ever formed).
//
// Work unit = (sample i, token tiles a' <= b' of 256 tokens), run by a pair
// of CTAs (a cluster of two, one tcgen05.mma.cta_group::2 per 16 features):
// CTA rank r stages tokens [256 a' + 128 r, +128) of A (then G) as the M
// half and tokens [256 b' + 128 r, +128) as the N half of the operands, and
// its TMEM holds rows 256 a' + 128 r .. of X = A_a' A_b'^T (K = d, columns
// 0..255) and of Y = G_a' G_b'^T (K = p, columns 256..511).  Both operands
// are K-major TMA tiles with 128-byte swizzle; each SM stages 32 KB per 64
// features, within its shared-memory bandwidth next to the tensor core's
// reads.  The epilogue of CTA r forms sum(X o Y) over its two 128 x 128
// blocks (2a'+r, 2b'+h), weighted 2 above the diagonal (the mirrored block),
// 1 on it, 0 below, and writes one partial per unit, CTA and epilogue warp;
// the last CTA to finish adds the partials of each sample in a fixed order.
//
// Units are dealt round-robin (unit u to pair u mod G).  All units cost the
// same, so when their count is not a multiple of the grid the last round is
// only partly busy; the units of that last round are therefore cut along p
// into `tail_split` sub-units that each recompute X over all of d but only
// a slice of Y's K range.  Because sum(X o Y) is linear in Y, the sub-units'
// partial sums simply add up: no combine step is needed.
//
// Pipeline: the leader's (rank 0) `full` barrier counts both CTAs' loads;
// the MMA's completion is multicast to both CTAs' `empty` and `tfull`; each
// epilogue releases the accumulators on the leader's `tempty`.
//
// Roles (320 threads): warp 0 = TMA producer (both CTAs), warp 1 = MMA issuer
// (rank 0) and TMEM owner, warps 2..9 = epilogue.
#include "common.cuh"

namespace dpclip {
namespace {

constexpr int kStages = 6;
constexpr uint32_t kTileBytes = 128 * 128;   // 128 token rows x 128 B (one K block)
constexpr uint32_t kStageTx = 4 * kTileBytes;   // both CTAs' two tiles of one stage
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint16_t kPairMask = 0x3;

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint64_t tempty;
  uint32_t tmem;
  int abort_flag;
  int issued;
  int consumed;
  int mma_units;
  int is_last;
  float red[kSumSamples * (kThreads / 32)];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * 2 * kTileBytes + sizeof(Ctl);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// unit index within a sample -> (a', b'): for b' = 0, 1, ... the tiles
// a' = 0 .. b'.
__device__ __forceinline__ void pair_of(int pr, int& a, int& bb) {
  int col = 0;
  while (pr > col) {
    pr -= col + 1;
    ++col;
  }
  a = pr;
  bb = col;
}

// Work item g -> (sample, unit index within the sample, p-block range).
struct GhostItem {
  int i, pr, pb0, pb1;
};
__device__ __forceinline__ bool ghost_item(const GhostParams& p, int g, GhostItem& it) {
  int u;
  if (g < p.nfull) {
    u = g;
    it.pb0 = 0;
    it.pb1 = p.pblocks;
  } else {
    const int t = g - p.nfull;
    if (t >= (p.B * p.npairs - p.nfull) * p.tail_split) return false;
    u = p.nfull + t / p.tail_split;
    const int c = t % p.tail_split;
    it.pb0 = c * p.pb_per_split;
    it.pb1 = min(it.pb0 + p.pb_per_split, p.pblocks);
  }
  it.i = u / p.npairs;
  it.pr = u % p.npairs;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) ghost_kernel(const __grid_constant__ GhostParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sP = smem;                              // this CTA's 128 tokens of tile a'
  uint8_t* sQ = sP + kStages * kTileBytes;         // its 128 tokens of tile b'
  Ctl* ctl = reinterpret_cast<Ctl*>(sQ + kStages * kTileBytes);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // clusters of (2, 1, 1) over a 1-D grid: CTA x is rank x % 2 of cluster x / 2
  const int rank = (int)(blockIdx.x & 1u);
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  if (cluster_nctarank() != 2u || cluster_ctarank() != (uint32_t)rank) {
    // not launched as clusters of two: nothing of the pair protocol may run
    if (threadIdx.x == 0) record_error(p.err, DPCLIP_ERR_CUDA);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull, 1);
    mbar_init(&ctl->tempty, 2 * 32 * kEpiWarps);
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
  if (warp == 1) tmem_alloc_pair(&ctl->tmem, 512);
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either uses the other's
  tc_fence_after();
  pdl_wait();   // inputs may come from the previous kernel
  const uint32_t tmem = ctl->tmem;
  const WaitCtx wc{&ctl->abort_flag, p.err, kWaitLimitNs};

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&ctl->full[0]), 0);   // the leader's
      int it = 0;
      bool run = true;
      GhostItem itm;
      for (int g = pair; run && ghost_item(p, g, itm); g += npairs) {
        const int i = itm.i;
        int a, b;
        pair_of(itm.pr, a, b);
        const int ta = (2 * a + rank) * kGhostTile, tb = (2 * b + rank) * kGhostTile;
        const int kblocks = p.dblocks + (itm.pb1 - itm.pb0);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) {
            run = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&ctl->full[s], kStageTx);
          const uint32_t bar = full0 + (uint32_t)s * (uint32_t)sizeof(uint64_t);
          const bool on_a = kb < p.dblocks;
          const CUtensorMap* map = on_a ? &p.map_a : &p.map_g;
          const int k0 = (on_a ? kb : itm.pb0 + kb - p.dblocks) * kBlockK;
          tma_load_3d_pair(sP + s * kTileBytes, map, bar, k0, ta, i);
          tma_load_3d_pair(sQ + s * kTileBytes, map, bar, k0, tb, i);
          ctl->issued = it + 1;
        }
      }
      // producer tail: the MMA's release of every stage this CTA filled has
      // arrived before the CTA may exit
      if (run)
        for (int j = it; j < it + kStages; ++j)
          if (!mbar_wait(&ctl->empty[j % kStages], ((j / kStages) & 1) ^ 1, wc)) break;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256, false, false);
      int it = 0, lu = 0;
      bool run = true;
      GhostItem itm;
      for (int g = pair; run && ghost_item(p, g, itm); g += npairs, ++lu) {
        if (!mbar_wait_cluster(&ctl->tempty, (lu & 1) ^ 1, wc)) {
          run = false;
          break;
        }
        tc_fence_after();
        const int kblocks = p.dblocks + (itm.pb1 - itm.pb0);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->full[s], (it / kStages) & 1, wc)) {
            run = false;
            break;
          }
          ctl->consumed = it + 1;
          tc_fence_after();
          const bool on_a = kb < p.dblocks;
          const int kl = on_a ? kb : kb - p.dblocks;
          const uint32_t dt = tmem + (on_a ? 0u : 256u);
          const uint32_t a0 = smem_u32(sP + s * kTileBytes);
          const uint32_t b0 = smem_u32(sQ + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_pair(dt, sdesc_sw128(a0 + kk * 32, 16, 1024),
                           sdesc_sw128(b0 + kk * 32, 16, 1024), idesc, (kl | kk) != 0);
          umma_commit_pair(&ctl->empty[s], kPairMask);
        }
        if (!run) break;
        umma_commit_pair(&ctl->tfull, kPairMask);
        ctl->mma_units = lu + 1;
      }
      // accumulator tail: both epilogues have released the accumulators
      // (their arrivals target this CTA)
      if (run) mbar_wait_cluster(&ctl->tempty, (lu & 1) ^ 1, wc);
    }
  } else {
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const uint32_t release = mapa_shared(smem_u32(&ctl->tempty), 0);
    int lu = 0;
    GhostItem itm;
    for (int g = pair; ghost_item(p, g, itm); g += npairs, ++lu) {
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->tfull, lu & 1, wc))) break;
      tc_fence_after();
      int aa, bb;
      pair_of(itm.pr, aa, bb);
      const int a = 2 * aa + rank;                   // 128-token block of these rows
      const int b = 2 * bb + half;                   // 128-token block of these columns
      const float w = a < b ? 2.f : (a == b ? 1.f : 0.f);
      const uint32_t base = tmem + (uint32_t)half * 128u + ((uint32_t)(quad * 32) << 16);
      float s = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float x[32], y[32];
        tmem_ld32(base + c4 * 32, x);
        tmem_ld32(base + 256 + c4 * 32, y);
#pragma unroll
        for (int j = 0; j < 32; ++j) s = fmaf(x[j], y[j], s);
      }
      tc_fence_before();
      mbar_arrive_remote(release);
      s = warp_sum(s);
      if (lane == 0) p.part[((size_t)g * 2 + rank) * kEpiWarps + ew] = w * s;
    }
  }

  // per sample: its whole units [i*np, (i+1)*np) below nfull, then the
  // sub-units of its units above nfull (item order = sample order); each
  // item has 2 * kEpiWarps partials (CTA rank, epilogue warp)
  {
    constexpr int kPer = 2 * kEpiWarps;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();   // the CTA's partials, written before the barrier
      ctl->is_last = atomic_add_acq_rel(p.ticket, 1u) == gridDim.x - 1u ? 1 : 0;
    }
    __syncthreads();
    if (ctl->is_last) {
      const int np = p.npairs, nf = p.nfull, ts = p.tail_split;
      auto f0 = [&](int i) { return min(i * np, nf); };
      auto s0 = [&](int i) { return nf + (max(i * np, nf) - nf) * ts; };
      auto n1 = [&](int i) { return (long long)(min((i + 1) * np, nf) - f0(i)) * kPer; };
      auto n2 = [&](int i) {
        return (long long)(nf + (max((i + 1) * np, nf) - nf) * ts - s0(i)) * kPer;
      };
      sum_per_sample(
          p.B, [&](int i) { return n1(i) + n2(i); },
          [&](int i, long long e) {
            const long long a = n1(i);
            return e < a ? p.part + (size_t)f0(i) * kPer + e : p.part + (size_t)s0(i) * kPer + (e - a);
          },
          1.f, p.sq, false, ctl->red, (int)threadIdx.x, kThreads, [] { __syncthreads(); });
      if (threadIdx.x == 0) *p.ticket = 0u;
    }
  }

  tc_fence_before();
  cluster_sync_all();   // every role of both CTAs has finished issuing
  if (threadIdx.x == 0) {
    // after a timeout in either CTA: let the loads and MMAs still in flight
    // (which may target the other CTA's barriers) land, boundedly
    uint32_t peer_flag;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(peer_flag)
                 : "r"(mapa_shared(smem_u32(&ctl->abort_flag), (uint32_t)(rank ^ 1)))
                 : "memory");
    if (ctl->abort_flag || peer_flag) {
      const uint64_t lim = 100000000ull;
      if (rank == 0) {
        for (int it = ctl->consumed; it < ctl->issued; ++it) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&ctl->full[it % kStages], (uint32_t)(it / kStages) & 1u))
            if (globaltimer_ns() - t0 > lim) break;
        }
        if (ctl->mma_units > 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&ctl->tfull, (uint32_t)(ctl->mma_units - 1) & 1u))
            if (globaltimer_ns() - t0 > lim) break;
        }
      }
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 10000000ull) {
      }
    }
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

size_t ghost_smem() { return kSmemBytes; }

// Tail split for `grid` pairs.
void plan_ghost_schedule(GhostParams& p, int grid) {
  const int units = p.B * p.npairs;
  const int rounds = units / grid;
  p.nfull = rounds * grid;
  const int tail = units - p.nfull;
  p.tail_split = 1;
  p.pb_per_split = p.pblocks;
  if (tail == 0) return;
  // cost of the last round in K-blocks; a unit is dblocks + pblocks
  double best = (double)p.dblocks + p.pblocks;
  for (int want = 2; want <= 8; ++want) {
    const int pbc = (p.pblocks + want - 1) / want;
    const int s = (p.pblocks + pbc - 1) / pbc;   // no empty slice
    const int extra_rounds = (tail * s + grid - 1) / grid;
    const double cost = (double)extra_rounds * (p.dblocks + pbc);
    if (cost < best - 1e-9) {
      best = cost;
      p.tail_split = s;
      p.pb_per_split = pbc;
    }
  }
}

cudaError_t launch_ghost(const GhostParams& params, cudaStream_t s) {
  GhostParams p = params;
  cudaError_t e = cudaFuncSetAttribute(ghost_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int resident =
      max_resident_pairs(reinterpret_cast<const void*>(ghost_kernel), kThreads, kSmemBytes, 3);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int pairs = std::max(1, std::min({resident, kMaxPersistentGrid / 2, p.B * p.npairs}));
  plan_ghost_schedule(p, pairs);
  return launch_pdl(ghost_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, s, 2, p);
}

}  // namespace dpclip
