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
//               (A_i^T G_i)^2.  The stored variant also writes every tile
//               to M_i = A_i^T G_i ([B][d][p] fp32): the clipped sum is then
//               an elementwise pass over M instead of a second GEMM.
//
// The tensor cores of two SMs work as a pair (a cluster of two CTAs, one
// tcgen05.mma.cta_group::2 per 16 tokens): a pair tile is 256 d-rows x 256
// p-columns.  CTA rank r loads, by TMA with 128-byte swizzle, its own 128
// d-columns of A and p-columns [128 r, 128 r + 128) of the tile from G (both
// operands MN-major: tokens are the slow axis of A and G), and holds rows
// [128 r, 128 r + 128) of the product in its TMEM.  Each SM thus stages 32 KB
// per 64 tokens instead of the 48 KB a one-CTA 128 x 256 tile needs, which
// keeps shared-memory traffic (TMA writes plus tensor-core reads) within its
// bandwidth.  A work item is (pair tile, sample i, a range of that sample's
// 64-token K-blocks); its accumulator lives in TMEM (256 columns) and two
// accumulators alternate, so the epilogue of one item overlaps the mainloop
// of the next.  Both CTAs of a pair walk the same item sequence; everything
// after the MMA (sums of squares, stores, tail tickets) is per CTA, on its
// own 128-row half ("CTA tile" = pair tile * 2 + rank).
//
// Item sequences of a pair (cluster c of G):
//   norm mode: items are whole (pair tile, sample) units dealt one by one,
//     sample-major (u = i * ntiles + tile; pair c takes u = c, c + G, ...),
//     so the pairs running together share one sample's A and G slabs in L2.
//   grad mode: `waves` full waves of whole tiles (pair c owns tiles c,
//     c + G, ...: all B samples of a tile, folded into a register running
//     sum s_0 acc_0 + s_1 acc_1 + ... in fp32), and the `ntail` remaining
//     tiles cut into lockstep bands of their time lines (the samples'
//     K-blocks one after another; grad_tail.cuh): each pair holds a few
//     segments (tile, K-block range), cut into items where a segment passes
//     from one sample to the next.  A CTA writes each partial half-tile to
//     the workspace slot of its segment, takes an integer ticket on its CTA
//     tile, and the last CTA to arrive adds the slots of the CTA tile in the
//     schedule's order (a fixed order), adds the noise and stores.  No CTA
//     ever waits on another pair.  Each pair runs its segments first: the
//     partial tiles are then combined while the tensor cores work through
//     the waves, and the kernel ends on whole tiles.
//     The finished block leaves through a per-warp staging tile; the noise is
//     drawn there, one Philox block of four columns per lane (store_block).
//
// Pipeline: the leader's `full` barrier of a stage counts the bytes of both
// CTAs' loads; the MMA's completion is multicast to the `empty` barriers of
// both CTAs and to both CTAs' `tfull`; each CTA's epilogue releases an
// accumulator by arriving on the leader's `tempty`.
//
// Roles (384 threads, three warpgroups): warp 0 = TMA producer (both CTAs),
// warp 1 = MMA issuer (rank 0) and TMEM owner, warps 2-3 idle; warps 4..11 =
// epilogue (warp w reads TMEM lanes 32*(w%4).., columns 128*((w-4)/4)..).
// The grad epilogue keeps a 128-float running sum per thread, so registers
// move from the first warpgroup to the epilogue warpgroups (setmaxnreg: 40
// and 232 per thread, which adds up to the 168 per thread the block is
// launched with; the host checks the compiled count before every launch).
#include <atomic>

#include "common.cuh"
#include "grad_tail.cuh"

namespace dpclip {
namespace {

constexpr int kStages = 6;
constexpr uint32_t kBox = 64 * 128;              // 64 tokens x 128 B (64 bf16)
constexpr uint32_t kABytes = 2 * kBox;           // this CTA's 128 d-columns
constexpr uint32_t kGBytes = 2 * kBox;           // this CTA's 128 of the tile's 256 p-columns
constexpr uint32_t kStageTx = 2 * (kABytes + kGBytes);   // both CTAs' loads of one stage
constexpr uint16_t kPairMask = 0x3;              // both CTAs of the cluster
constexpr int kThreads = 128 + 32 * kEpiWarps;   // 384: producer warpgroup + 2 epilogue
constexpr int kEpiThreads = 32 * kEpiWarps;      // 256
constexpr int kEpiWarp0 = 4;                     // first epilogue warp
constexpr int kRegsProducer = 40;                // setmaxnreg shares (per thread)
constexpr int kRegsEpilogue = 232;
constexpr int kRegsAtLaunch = 168;               // needed: 128*40 + 256*232 <= 384*168
static_assert(128 * kRegsProducer + kEpiThreads * kRegsEpilogue <= kThreads * kRegsAtLaunch,
              "register split exceeds the block's allocation");

// A tail segment of this pair as its items see it: samples i0..i1, the
// first item from K-block kb0, the last up to kb1.
struct PairSeg {
  int tile, slot, i0, i1, kb0, kb1, whole, pad;
};

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem;
  int abort_flag;
  int issued;
  int consumed;
  int mma_units;     // items whose MMAs were committed to tfull
  int is_last;
  int combine;
  int nseg;          // grad mode: this pair's tail segments
  PairSeg seg[kTailMaxSegs];
  float red[kThreads / 32];
};

static_assert(sizeof(Ctl) % 16 == 0, "staging tiles after Ctl must be 16-byte aligned");
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * (kABytes + kGBytes) + sizeof(Ctl);
// Stored norm mode: one 32 x 33 fp32 transpose tile per epilogue warp, so
// that each store instruction writes 32 consecutive floats of one row.
constexpr size_t kStoreTileFloats = 32 * 33;
constexpr size_t kSmemBytesStore = kSmemBytes + kEpiWarps * kStoreTileFloats * sizeof(float);
static_assert(kSmemBytesStore <= 232448, "stored variant exceeds the shared memory of a CTA");
// Grad mode: one 32-row x 16-column fp32 staging tile per epilogue warp (four
// 16-byte blocks per row, their order swizzled by row so that both the
// row-per-thread writes and the block-per-lane reads are free of bank
// conflicts).
constexpr size_t kGradTileFloats = 32 * 16;
constexpr size_t kSmemBytesGrad = kSmemBytes + kEpiWarps * kGradTileFloats * sizeof(float);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float clip_scale(float q, float C) {
  return q > 0.f ? fminf(1.f, C / sqrtf(q)) : 1.f;
}

// Barrier among the 256 epilogue threads only (named barrier 1).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// Same barrier, returning true iff `ok` holds in every epilogue thread (keeps
// the epilogue warps in step when one of them gives up on a wait).
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

struct Item {
  int tile, i, kb0, kb1;   // tile: pair tile
  int slot;         // tail segment: its workspace slot (pair level)
  bool seg_first;   // first item of this pair's part of the tile: reset the sum
  bool seg_last;    // last item of this pair's part of the tile: finish it
  bool whole;       // this pair holds every item of the tile
};

// Position of this pair in the grid of pairs.
struct PairPos {
  int c, G;   // cluster index, number of clusters
};

// The k-th item of this pair; false past the end.  `seg` holds the pair's
// tail segments (grad mode), found once at the start of the kernel.
template <bool kGrad>
__device__ __forceinline__ bool item_at(const GemmDpParams& p, const PairPos& pp,
                                        const PairSeg* seg, int nseg, int k, Item& it) {
  const int G = pp.G, c = pp.c, B = p.B;
  const int ntiles = (p.mtiles >> 1) * p.ntiles;
  if constexpr (!kGrad) {
    const long long u = (long long)c + (long long)k * G;
    if (u >= (long long)ntiles * B) return false;
    it.i = (int)(u / ntiles);
    it.tile = (int)(u % ntiles);
    it.kb0 = 0;
    it.kb1 = p.tblocks;
    it.slot = -1;
    it.seg_first = it.seg_last = it.whole = true;
    return true;
  } else {
    // first this pair's segments of the tail tiles (each cut where the time
    // line passes from one sample to the next), so that the partial tiles are
    // combined while the tensor cores run the full waves; then the waves
    for (int j = 0; j < nseg; ++j) {
      const PairSeg sg = seg[j];
      if (k <= sg.i1 - sg.i0) {
        it.tile = p.waves * G + sg.tile;
        it.i = sg.i0 + k;
        it.kb0 = k == 0 ? sg.kb0 : 0;
        it.kb1 = it.i == sg.i1 ? sg.kb1 : p.tblocks;
        it.slot = sg.slot;
        it.seg_first = k == 0;
        it.seg_last = it.i == sg.i1;
        it.whole = sg.whole != 0;
        return true;
      }
      k -= sg.i1 - sg.i0 + 1;
    }
    if (k >= p.waves * B) return false;
    it.tile = c + (k / B) * G;
    it.i = k % B;
    it.kb0 = 0;
    it.kb1 = p.tblocks;
    it.slot = -1;
    it.seg_first = it.i == 0;
    it.seg_last = it.i == B - 1;
    it.whole = true;
    return true;
  }
}

// Finishes the warp's 32 x 128 block of the gradient: lane l holds, in tot,
// columns cb .. cb+127 of row r0 + l.  Per 16-column chunk the rows go
// through the staging tile; lane l then takes row 8g + l / 4 (g = 0..3) and
// the 16-byte block l % 4 of the chunk, adds sigma C z from that block's
// Philox draw (the gradient's row-major blocks of four: (r p + c) / 4), and
// writes it (rows beyond d and columns beyond p skipped; p is a multiple of
// 8), with the fused update theta -= (lr / L) g when asked.  The loop over
// rows stays rolled, so one copy of the generator serves every block.
__device__ __forceinline__ void store_block(const GemmDpParams& p, int r0, int cb,
                                            const float (&tot)[128], float4* tb) {
  const int lane = threadIdx.x & 31;
  const float nscale = p.sigma * p.C;
  const int nrows = min(32, p.d - r0);
  const int swz = (lane >> 1) & 3;
#pragma unroll 1
  for (int ch = 0; ch < 8; ++ch) {
    __syncwarp();
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) {
      if (q8 == ch) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tb[lane * 4 + (q ^ swz)] = make_float4(tot[16 * q8 + 4 * q], tot[16 * q8 + 4 * q + 1],
                                                 tot[16 * q8 + 4 * q + 2], tot[16 * q8 + 4 * q + 3]);
      }
    }
    __syncwarp();
    const int c = cb + 16 * ch + 4 * (lane & 3);
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      const int rl = 8 * g + (lane >> 2);
      float4 v = tb[rl * 4 + ((lane & 3) ^ ((rl >> 1) & 3))];
      if (rl < nrows && c < p.p) {
        const size_t e = (size_t)(r0 + rl) * p.p + c;
        if (nscale != 0.f) {
          float z[4];
          philox_normal4_fast(p.seed, 3u, p.offset, (uint32_t)(e >> 2), z);
          v.x = fmaf(nscale, z[0], v.x);
          v.y = fmaf(nscale, z[1], v.y);
          v.z = fmaf(nscale, z[2], v.z);
          v.w = fmaf(nscale, z[3], v.w);
        }
        if (p.grad) *reinterpret_cast<float4*>(p.grad + e) = v;
        if (p.upd_param) {
          float4 w = *reinterpret_cast<const float4*>(p.upd_param + e);
          w.x = fmaf(-p.upd_scale, v.x, w.x);
          w.y = fmaf(-p.upd_scale, v.y, w.y);
          w.z = fmaf(-p.upd_scale, v.z, w.z);
          w.w = fmaf(-p.upd_scale, v.w, w.w);
          *reinterpret_cast<float4*>(p.upd_param + e) = w;
        }
      }
    }
  }
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
  // clusters of (2, 1, 1) over a 1-D grid: CTA x is rank x % 2 of cluster x / 2
  const int rank = (int)(blockIdx.x & 1u);
  const PairPos pp{(int)(blockIdx.x >> 1), (int)(gridDim.x >> 1)};
  const int mp = p.mtiles >> 1;   // pair tiles along d
  const int ntiles_cta = p.mtiles * p.ntiles;
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
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 2 * kEpiThreads);
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
  if (warp == 1) tmem_alloc_pair(&ctl->tmem, 512);
  if (kGrad && threadIdx.x == 64) {
    // this pair's tail segments (the host keeps them within kTailMaxSegs)
    TailSeg sgs[kTailMaxSegs];
    const int ns = tail_pair_segs(pp.G, p.ntail, (long long)p.B * p.tblocks, p.tail_cover, pp.c, sgs);
    for (int j = 0; j < ns; ++j) {
      const TailSeg& sg = sgs[j];
      PairSeg& q = ctl->seg[j];
      q.tile = sg.tile;
      q.slot = sg.slot;
      q.i0 = (int)(sg.t0 / p.tblocks);
      q.i1 = (int)((sg.t1 - 1) / p.tblocks);
      q.kb0 = (int)(sg.t0 - (long long)q.i0 * p.tblocks);
      q.kb1 = (int)(sg.t1 - (long long)q.i1 * p.tblocks);
      q.whole = sg.t0 == 0 && sg.t1 == (long long)p.B * p.tblocks;
    }
    ctl->nseg = ns;
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either uses the other's
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
  const int nseg = kGrad ? ctl->nseg : 0;
  const WaitCtx wc{&ctl->abort_flag, p.err, kWaitLimitNs};
  if (warp < kEpiWarp0) {
    regs_dec<kRegsProducer>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&ctl->full[0]), 0);   // the leader's
      int it = 0;
      Item itm;
      bool run = true;
      for (int k = 0; run && item_at<kGrad>(p, pp, ctl->seg, nseg, k, itm); ++k) {
        const int d0 = (2 * (itm.tile % mp) + rank) * kDpTileM;
        const int p0 = (itm.tile / mp) * kDpTileN + rank * (kDpTileN / 2);
        for (int kb = itm.kb0; kb < itm.kb1; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1, wc)) {
            run = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&ctl->full[s], kStageTx);
          const uint32_t bar = full0 + (uint32_t)s * (uint32_t)sizeof(uint64_t);
          const int t0 = kb * 64;
          uint8_t* a = sA + s * kABytes;
          uint8_t* g = sG + s * kGBytes;
          tma_load_3d_pair(a, &p.map_a, bar, d0, t0, itm.i);
          tma_load_3d_pair(a + kBox, &p.map_a, bar, d0 + 64, t0, itm.i);
          tma_load_3d_pair(g, &p.map_g, bar, p0, t0, itm.i);
          tma_load_3d_pair(g + kBox, &p.map_g, bar, p0 + 64, t0, itm.i);
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
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(256, kDpTileN, true, true);
      int it = 0, u = 0;
      Item itm;
      bool run = true;
      for (; run && item_at<kGrad>(p, pp, ctl->seg, nseg, u, itm); ++u) {
        const int acc = u & 1;
        if (!mbar_wait_cluster(&ctl->tempty[acc], ((u >> 1) & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)acc * 256u;
        for (int kb = itm.kb0; kb < itm.kb1; ++kb, ++it) {
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
            umma_bf16_pair(dt, sdesc_sw128(a0 + kk * 2048, kBox, 1024),
                           sdesc_sw128(g0 + kk * 2048, kBox, 1024), idesc,
                           (kb != itm.kb0 || kk != 0) ? 1u : 0u);
          }
          umma_commit_pair(&ctl->empty[s], kPairMask);
        }
        if (!run) break;
        umma_commit_pair(&ctl->tfull[acc], kPairMask);
        ctl->mma_units = u + 1;
      }
      // accumulator tail: both epilogues have released every accumulator
      // (their arrivals target this CTA)
      if (run)
        for (int v = u; v < u + 2; ++v)
          if (!mbar_wait_cluster(&ctl->tempty[v & 1], ((v >> 1) & 1) ^ 1, wc)) break;
    }
  }
  } else {
    regs_inc<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int etid = ew * 32 + lane;   // 0..255, same role in every CTA
    const uint32_t tempty0 = mapa_shared(smem_u32(&ctl->tempty[0]), 0);
    float tot[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) tot[j] = 0.f;
    Item itm;
    for (int u = 0; item_at<kGrad>(p, pp, ctl->seg, nseg, u, itm); ++u) {
      const int acc = u & 1;
      if (!epi_all(mbar_wait(&ctl->tfull[acc], (u >> 1) & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem + (uint32_t)acc * 256u + (uint32_t)half * 128u + ((uint32_t)(quad * 32) << 16);
      const uint32_t release = tempty0 + (uint32_t)acc * (uint32_t)sizeof(uint64_t);
      const int ctile = 2 * itm.tile + rank;                     // this CTA's tile
      const int row0 = (2 * (itm.tile % mp) + rank) * kDpTileM;  // its first d-row
      const int col0 = (itm.tile / mp) * kDpTileN;               // the tile's first p-column
      if (kGrad) {
        const float si = clip_scale(p.sqnorms[itm.i], p.C);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float v[32];
          tmem_ld32(taddr + c4 * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            tot[c4 * 32 + j] = itm.seg_first ? si * v[j] : fmaf(si, v[j], tot[c4 * 32 + j]);
        }
        tc_fence_before();
        mbar_arrive_remote(release);
        bool do_store = false;
        if (itm.seg_last) {
          do_store = itm.whole;
          if (!itm.whole) {
            // partial tile: publish this CTA's part; the last CTA to arrive
            // on the CTA tile adds every participant's part, in the order of
            // the schedule, and stores
            const int tt = itm.tile - p.waves * pp.G;
            const long long L = (long long)p.B * p.tblocks;
            float4* slot = reinterpret_cast<float4*>(p.slots) +
                           (size_t)(2 * itm.slot + rank) * (32 * kEpiThreads);
#pragma unroll
            for (int jb = 0; jb < 32; ++jb)
              __stcg(slot + jb * kEpiThreads + etid,
                     make_float4(tot[4 * jb], tot[4 * jb + 1], tot[4 * jb + 2], tot[4 * jb + 3]));
            __threadfence();
            epi_sync();
            if (etid == 0) {
              int parts = 0;
              tail_tile_slots(pp.G, p.ntail, L, p.tail_cover, tt, [&](int) { ++parts; });
              const uint32_t prev = atomicAdd(&p.tickets[ctile], 1u);
              ctl->combine = prev == (uint32_t)(parts - 1);
            }
            epi_sync();
            if (ctl->combine) {
              __threadfence();
#pragma unroll
              for (int j = 0; j < 128; ++j) tot[j] = 0.f;
              tail_tile_slots(pp.G, p.ntail, L, p.tail_cover, tt, [&](int sl) {
                const float4* src = reinterpret_cast<const float4*>(p.slots) +
                                    (size_t)(2 * sl + rank) * (32 * kEpiThreads);
#pragma unroll
                for (int jb = 0; jb < 32; ++jb) {
                  const float4 v = __ldcg(src + jb * kEpiThreads + etid);
                  tot[4 * jb] += v.x;
                  tot[4 * jb + 1] += v.y;
                  tot[4 * jb + 2] += v.z;
                  tot[4 * jb + 3] += v.w;
                }
              });
              do_store = true;
            }
          }
        }
        if (do_store && row0 + quad * 32 < p.d)
          store_block(p, row0 + quad * 32, col0 + half * 128, tot,
                      reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(ctl) + sizeof(Ctl)) +
                          (size_t)ew * (kGradTileFloats / 4));
      } else {
        float ss = 0.f;
        if (p.pstore) {
          // stored variant: read the whole 32 x 128 slab, release the
          // accumulator, then write the slab to M_i through a per-warp
          // transpose tile, one 128-byte row segment per store instruction
          float v[4][32];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(taddr + c4 * 32, v[c4]);
          tc_fence_before();
          mbar_arrive_remote(release);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(v[c4][j], v[c4][j], ss);
          float* tb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ctl) + sizeof(Ctl)) +
                      (size_t)ew * kStoreTileFloats;
          const int r0 = row0 + quad * 32;
          const int cb = col0 + half * 128;
          const int nrows = min(32, p.d - r0);
          float* mbase = p.pstore + ((size_t)itm.i * p.d + r0) * p.p;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; ++j) tb[lane * 33 + j] = v[c4][j];
            __syncwarp();
            const int c = cb + c4 * 32 + lane;
            if (c < p.p)
              for (int rr = 0; rr < nrows; ++rr) mbase[(size_t)rr * p.p + c] = tb[rr * 33 + lane];
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float v[32];
            tmem_ld32(taddr + c4 * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
          }
          tc_fence_before();
          mbar_arrive_remote(release);
        }
        ss = warp_sum(ss);
        if (lane == 0) p.part[((size_t)ctile * p.B + itm.i) * kEpiWarps + ew] = ss;
      }
    }
  }

  if (!kGrad)
    reduce_partials_last_cta(p.part, p.B, ntiles_cta, p.B, 1, kEpiWarps, 1.f, p.sq, p.ticket,
                             ctl->red, &ctl->is_last, p.accumulate != 0);

  tc_fence_before();
  cluster_sync_all();   // every role of both CTAs has finished issuing
  // after a timeout in either CTA: let the loads and MMAs still in flight
  // (which may target the other CTA's barriers) land, boundedly
  if (threadIdx.x == 0) {
    int any_abort = ctl->abort_flag;
    uint32_t peer_flag;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(peer_flag)
                 : "r"(mapa_shared(smem_u32(&ctl->abort_flag), (uint32_t)(rank ^ 1)))
                 : "memory");
    any_abort |= (int)peer_flag;
    if (any_abort) {
      const uint64_t lim = 100000000ull;
      if (rank == 0) {
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
      // arrivals multicast to this CTA, and the other CTA's loads, land
      // within microseconds of the work above
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

size_t gemm_dp_smem() { return kSmemBytes; }

size_t gemm_dp_slot_bytes(int max_grid) {
  // kTailMaxSegs contributions per pair, one half-tile slot per CTA each
  return (size_t)kTailMaxSegs * max_grid * 32 * kEpiThreads * 16;
}

TailStats grad_tail_stats(int G, int ntail, long long L, uint32_t cover) {
  TailStats st{};
  if (G < 1 || G > kMaxPersistentGrid / 2) return st;
  long long work[kMaxPersistentGrid / 2] = {};
  int segs[kMaxPersistentGrid / 2] = {};
  bool covered = false;
  TailWalk w;
  w.start(G, ntail, L, cover);
  while (!w.done) {
    ++st.levels;
    for (int c = w.p0; c < w.p0 + w.n; ++c) {
      TailSeg sg;
      if (tail_seg_of(w, c, sg) > 0 && sg.t1 > sg.t0) {
        work[c] += sg.t1 - sg.t0;
        ++segs[c];
        ++st.nsegs;
        st.nslots = std::max(st.nslots, sg.slot + 1);
      }
    }
    if (w.band() && w.cover) covered = true;
    w.advance(cover);
  }
  st.complete = covered || w.m == 0 || w.t1 <= w.t0;
  for (int c = 0; c < G; ++c) {
    st.max_work = std::max(st.max_work, work[c]);
    st.max_segs = std::max(st.max_segs, segs[c]);
  }
  return st;
}

void grad_tail_dump(int G, int ntail, long long L, uint32_t cover, int64_t* segs, int seg_cap,
                    int* nsegs, int64_t* contrib, int contrib_cap, int* ncontrib) {
  int ns = 0, nc = 0;
  for (int c = 0; c < G && ntail > 0; ++c) {
    // the segments of the kernel's prologue, for pair c
    TailSeg sgs[kTailMaxSegs];
    const int n = tail_pair_segs(G, ntail, L, cover, c, sgs);
    for (int j = 0; j < n; ++j, ++ns) {
      if (ns < seg_cap) {
        int64_t* o = segs + 5 * (size_t)ns;
        o[0] = c;
        o[1] = sgs[j].tile;
        o[2] = sgs[j].t0;
        o[3] = sgs[j].t1;
        o[4] = sgs[j].slot;
      }
    }
  }
  struct Emit {
    int64_t* out;
    int cap, tt;
    int* n;
    __host__ __device__ void operator()(int sl) const {
      if (*n < cap) {
        out[2 * (size_t)*n] = tt;
        out[2 * (size_t)*n + 1] = sl;
      }
      ++*n;
    }
  };
  for (int tt = 0; tt < ntail; ++tt)
    tail_tile_slots(G, ntail, L, cover, tt, Emit{contrib, contrib_cap, tt, &nc});
  *nsegs = ns;
  *ncontrib = nc;
}

// Grad-mode schedule over `grid` pairs: full waves of whole pair tiles (every
// pair works on the same sample at the same time, so pairs that share A and
// G slabs find them in L2), and the remaining tiles cut into lockstep bands
// (grad_tail.cuh).  Of the schedules that make the first k band levels exact
// and the next one cover, the one with the least work on its busiest pair
// is taken (then the fewest partial tiles), among those that keep every pair
// within kTailMaxSegs partial tiles; k = 0 (one cover level: q bands of the
// whole time line, the remaining pairs idle in the tail) always qualifies.
void plan_grad_schedule(int ntiles, int B, int tblocks, int grid, int& waves, int& ntail,
                        uint32_t& cover) {
  waves = ntiles / grid;
  ntail = ntiles - waves * grid;
  cover = ~0u;
  if (ntail == 0) return;
  // the last plan of this host thread (a training loop repeats its shapes)
  thread_local int key[4] = {-1, -1, -1, -1};
  thread_local uint32_t key_cover = ~0u;
  if (key[0] == ntiles && key[1] == B && key[2] == tblocks && key[3] == grid) {
    cover = key_cover;
    return;
  }
  const long long L = (long long)B * tblocks;
  long long best = -1, best_segs = 0;
  for (int k = 0; k < kTailMaxLevels; ++k) {
    const uint32_t mask = ~0u << k;
    const TailStats st = grad_tail_stats(grid, ntail, L, mask);
    if (st.complete && st.max_segs <= kTailMaxSegs && st.nslots <= kTailMaxSegs * grid &&
        (best < 0 || st.max_work < best || (st.max_work == best && st.nsegs < best_segs))) {
      best = st.max_work;
      best_segs = st.nsegs;
      cover = mask;
    }
    if (st.levels <= k) break;   // the walk ended before level k: larger k change nothing
  }
  key[0] = ntiles;
  key[1] = B;
  key[2] = tblocks;
  key[3] = grid;
  key_cover = cover;
}

// The register split above is only safe when the compiled kernel is launched
// with at least kRegsAtLaunch registers per thread.
template <typename K>
cudaError_t check_regs(K kernel) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  return fa.numRegs >= kRegsAtLaunch ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemm_dp(const GemmDpParams& params, bool grad_mode, cudaStream_t s) {
  GemmDpParams p = params;
  if (p.mtiles % 2 != 0) return cudaErrorInvalidValue;
  cudaError_t e;
  auto kernel = grad_mode ? gemm_dp_kernel<true> : gemm_dp_kernel<false>;
  if ((e = check_regs(kernel)) != cudaSuccess) return e;
  const size_t smem = grad_mode ? kSmemBytesGrad : (p.pstore ? kSmemBytesStore : kSmemBytes);
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  const int resident = max_resident_pairs(reinterpret_cast<const void*>(kernel), kThreads, smem,
                                          grad_mode ? 0 : (p.pstore ? 2 : 1));
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int ntiles = (p.mtiles / 2) * p.ntiles;   // pair tiles
  // one pair per two SMs, fewer when there is little work
  const long long work = (long long)ntiles * p.B * (grad_mode ? 4 : 1);
  long long pairs_ll = std::min((long long)resident, (long long)(kMaxPersistentGrid / 2));
  pairs_ll = std::max(1LL, std::min(pairs_ll, work));
  const int pairs = (int)pairs_ll;
  if (grad_mode)
    plan_grad_schedule(ntiles, p.B, p.tblocks, pairs, p.waves, p.ntail, p.tail_cover);
  return launch_pdl(kernel, dim3(2 * pairs), dim3(kThreads), smem, s, 2, p);
}

// Pairs (clusters of two CTAs, one per SM) of a kernel variant that can be
// resident at once, per device; `slot` names the variant for the cache
// (atomics: calls may come from several host threads).
int max_resident_pairs(const void* kernel, int threads, size_t smem, int slot) {
  static std::atomic<int> cache[16][kPairSlots];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) dev = 0;
  if (slot < 0 || slot >= kPairSlots) return 0;
  const int cached = cache[dev][slot].load(std::memory_order_relaxed);
  if (cached > 0) return cached;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxPersistentGrid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev][slot].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace dpclip
