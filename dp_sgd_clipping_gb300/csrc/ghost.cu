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
// into `tail_split` sub-units, each with a slice of Y's K range.  Because
// sum(X o Y) is linear in Y, the sub-units' partial sums simply add up.  X
// (K = d) is either recomputed by every sub-unit or, when each pair has at
// most one sub-unit of the last round (`tail_shared`), formed once by an
// extra X sub-unit that stores it (fp32, 256 KB per unit) for the Y
// sub-units: each epilogue warp of the X sub-unit releases a counter once
// its rows are stored, and the matching warp of every Y sub-unit (same CTA
// rank, same rows and columns) waits for that counter, bounded, before it
// reads them.  All pairs are resident (the grid is the resident count), so
// the X sub-unit always runs; its own pair never waits on the others.
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

// Work item g -> (sample, unit index within the sample, K ranges: the first
// kx K-blocks over d, then p-blocks [pb0, pb1)) and its role.
enum { kWhole = 0, kXOnly = 1, kYOnly = 2 };
struct GhostItem {
  int i, pr, pb0, pb1, kx, role, tu;
};
__device__ __forceinline__ bool ghost_item(const GhostParams& p, int g, GhostItem& it) {
  int u;
  it.kx = p.dblocks;
  it.role = kWhole;
  it.tu = 0;
  if (g < p.nfull) {
    u = g;
    it.pb0 = 0;
    it.pb1 = p.pblocks;
  } else {
    const int per = p.tail_split + p.tail_shared;
    const int t = g - p.nfull;
    if (t >= (p.B * p.npairs - p.nfull) * per) return false;
    it.tu = t / per;
    u = p.nfull + it.tu;
    int c = t % per;
    if (p.tail_shared) {
      if (c == 0) {
        it.role = kXOnly;
      } else {
        it.role = kYOnly;
        it.kx = 0;
      }
      c -= 1;
    }
    it.pb0 = c < 0 ? 0 : c * p.pb_per_split;
    it.pb1 = c < 0 ? 0 : min(it.pb0 + p.pb_per_split, p.pblocks);
  }
  it.i = u / p.npairs;
  it.pr = u % p.npairs;
  return true;
}

// Spins (bounded; also ends once the call has recorded an error) until the
// counter is nonzero; acquire ordering for the loads that follow it.
__device__ __forceinline__ void wait_ready(const uint32_t* c, uint32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v != 0u) return;
    if (*reinterpret_cast<volatile uint32_t*>(err) != 0u) return;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, DPCLIP_ERR_TIMEOUT);
      return;
    }
    __nanosleep(64);
  }
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
        const int kblocks = itm.kx + (itm.pb1 - itm.pb0);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) {
            run = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&ctl->full[s], kStageTx);
          const uint32_t bar = full0 + (uint32_t)s * (uint32_t)sizeof(uint64_t);
          const bool on_a = kb < itm.kx;
          const CUtensorMap* map = on_a ? &p.map_a : &p.map_g;
          const int k0 = (on_a ? kb : itm.pb0 + kb - itm.kx) * kBlockK;
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
        const int kblocks = itm.kx + (itm.pb1 - itm.pb0);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->full[s], (it / kStages) & 1, wc)) {
            run = false;
            break;
          }
          ctl->consumed = it + 1;
          tc_fence_after();
          const bool on_a = kb < itm.kx;
          const int kl = on_a ? kb : kb - itm.kx;
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
      // this thread's row of X (shared tail): [unit][rank][row][256 columns]
      const size_t xrow = (((size_t)itm.tu * 2 + rank) * 128 + quad * 32 + lane) * 256 + half * 128;
      const size_t xflag = ((size_t)itm.tu * 2 + rank) * kEpiWarps + ew;   // its warp's counter
      float s = 0.f;
      if (itm.role == kXOnly) {
        // store X for the Y sub-units of this unit, then release it
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float x[64];
          tmem_ld64(base + c2 * 64, x);
          float4* dst = reinterpret_cast<float4*>(p.xbuf + xrow + c2 * 64);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        }
        tc_fence_before();
        mbar_arrive_remote(release);
        __syncwarp();
        if (lane == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.xready + xflag) : "memory");
      } else {
        if (itm.role == kYOnly) {
          if (lane == 0) wait_ready(p.xready + xflag, p.err);
          __syncwarp();
        }
        // the accumulators are released only after these loads: one wait
        // per 64 columns of X and Y keeps the gap before the next unit short
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float x[64], y[64];
          if (itm.role == kYOnly) {
            tmem_ld64(base + 256 + c2 * 64, y);
            const float4* src = reinterpret_cast<const float4*>(p.xbuf + xrow + c2 * 64);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float4 v = __ldcg(src + j);
              x[4 * j] = v.x;
              x[4 * j + 1] = v.y;
              x[4 * j + 2] = v.z;
              x[4 * j + 3] = v.w;
            }
          } else {
            tmem_ld64x2(base + c2 * 64, x, base + 256 + c2 * 64, y);
          }
#pragma unroll
          for (int j = 0; j < 64; ++j) s = fmaf(x[j], y[j], s);
        }
        tc_fence_before();
        mbar_arrive_remote(release);
      }
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
      const int np = p.npairs, nf = p.nfull, ts = p.tail_split + p.tail_shared;
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

// Tail split for `grid` pairs: the cut of the last round's units that
// minimises that round's cost in K-blocks.  A unit is dblocks + pblocks.
// Recomputing X, a sub-unit costs dblocks + its p-slice.  Sharing X (only
// when every sub-unit of the round fits on its own pair, so that no pair
// both waits for an X and owes one) costs max(dblocks, p-slice) plus the
// store of X, the wait and its reload: about 3.3 us measured on the up_proj
// shape (a 12-unit tail: 385 -> 381.6 us where 22 K-blocks, 6.8 us, were
// saved), i.e. about 10 K-blocks of 0.31 us.
constexpr int kSharedXCost = 10;

void plan_ghost_schedule(GhostParams& p, int grid) {
  const int units = p.B * p.npairs;
  const int rounds = units / grid;
  p.nfull = rounds * grid;
  const int tail = units - p.nfull;
  p.tail_split = 1;
  p.pb_per_split = p.pblocks;
  p.tail_shared = 0;
  if (tail == 0) return;
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
  for (int want = 1; want <= 8; ++want) {
    const int pbc = (p.pblocks + want - 1) / want;
    const int s = (p.pblocks + pbc - 1) / pbc;
    if (tail * (s + 1) > grid) break;
    const double cost = (double)std::max(p.dblocks, pbc) + kSharedXCost;
    if (cost < best - 1e-9) {
      best = cost;
      p.tail_split = s;
      p.pb_per_split = pbc;
      p.tail_shared = 1;
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
