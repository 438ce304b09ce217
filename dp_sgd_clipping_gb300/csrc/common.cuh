// Device-side building blocks shared by the dpclip kernels (sm_103a only):
// bounded mbarrier waits, TMA tile loads, tcgen05 (TMEM allocation, MMA,
// commit, loads), shared-memory / instruction descriptors, Philox-4x32-10 and
// the Box-Muller map, bf16 hi/lo splitting and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dpclip {

// ---------------------------------------------------------------------------
// Error word and bounded waits
// ---------------------------------------------------------------------------

// A device-side wait gives up after this long (ns of %globaltimer) unless the
// launch asks for a different limit.  Every kernel finishes in milliseconds.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Records `code` in the workspace error word (first writer wins).
__device__ __forceinline__ void record_error(uint32_t* err, int code) {
  if (err) atomicCAS(err, 0u, (uint32_t)code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes initialised barriers visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Per-CTA abort flag lives in shared memory; once any role of the CTA gives
// up, every other wait of the CTA returns false at once.
struct WaitCtx {
  volatile int* abort;   // shared memory flag
  uint32_t* err;         // workspace error word (global)
  uint64_t limit_ns;
};

// Waits for the phase with parity `parity` of `bar`.  Returns false when the
// CTA aborted or the limit expired (then the CTA is marked aborted and
// DPCLIP_ERR_TIMEOUT recorded).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if ((++n & 15u) == 0 && globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      record_error(w.err, DPCLIP_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel allows the next kernel of the
// stream to be scheduled as soon as all of its CTAs are running
// (pdl_trigger), and reads or writes global memory only after pdl_wait,
// which returns once the previous kernel has completed and its writes are
// visible.  Both are no-ops for launches without the attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  Coordinates are element indices, innermost
// first; out-of-range elements are filled with zeros.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// An L2 policy that evicts the lines a load brings in first: for an operand
// streamed once, so that it does not push out data that is read again.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_3d with an L2 eviction policy (l2_evict_first_policy).
__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, int c2,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------

// Whole-warp call: allocates `ncols` TMEM columns (power of two >= 32) and
// writes the base address to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its own TMEM
// lane (lane = 32 * (warp % 4) + lane id, encoded in taddr's upper half).
// One load of 64 consecutive fp32 columns and its wait, as in tmem_ld32.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

// Two loads of 64 consecutive fp32 columns each (one at taddr_a, one at
// taddr_b) behind a single wait: each thread gets its own TMEM lane's
// columns, as in tmem_ld32.
__device__ __forceinline__ void tmem_ld64x2(uint32_t taddr_a, float (&a)[64], uint32_t taddr_b,
                                            float (&b)[64]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr_a), "r"(taddr_b)
      : "memory");
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    a[j] = __uint_as_float(r[j]);
    b[j] = __uint_as_float(r[64 + j]);
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ---------------------------------------------------------------------------
// CTA pairs: a thread-block cluster of two CTAs whose tensor cores run one
// tcgen05.mma.cta_group::2 together.  CTA rank 0 of the pair issues the MMAs;
// operand A is split by rows (M) and B by columns (N) between the two CTAs'
// shared memory, and each CTA's TMEM holds its own M/2 rows of the product.
// Every tcgen05 instruction of a kernel that uses pairs says cta_group::2.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Address, in the cluster's shared-memory window, of the variable at this
// CTA's shared address `saddr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// atomicAdd with release and acquire semantics at GPU scope: the caller's
// earlier writes are visible before the increment, and after it the caller
// (and, past a CTA barrier, its CTA) sees what the earlier incrementers
// wrote before theirs.  One round trip instead of a fence and an atomic.
__device__ __forceinline__ uint32_t atomic_add_acq_rel(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

// 16 bytes into the shared memory of a CTA of the cluster (address from
// mapa_shared, 16-byte aligned).  A posted store: a later cluster barrier
// (release / acquire) makes it visible to that CTA.
__device__ __forceinline__ void st_dsmem_v4(uint32_t caddr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// All threads of all CTAs of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its cluster-window address (possibly in the
// other CTA of the pair).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// mbar_wait for a barrier that receives arrivals from the other CTA.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const WaitCtx& w) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*w.abort) return false;
    if ((++n & 15u) == 0 && globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      record_error(w.err, DPCLIP_ERR_TIMEOUT);
      return false;
    }
  }
}

// 3-D tiled load into this CTA's shared memory whose completion is counted
// on a barrier of either CTA of the pair (cluster-window address).
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Whole-warp calls, made by one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (+)= A * B over the pair (issued by rank 0 only); bf16 in, fp32 out.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at this shared address in every CTA of
// `cta_mask` when the MMAs issued so far complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Register reallocation between warpgroups (all threads of a warpgroup
// execute it): dec gives registers back, inc takes them, up to the block's
// launch allocation.
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// 1024-byte swizzle atoms start on 1024-byte boundaries.
//   K-major operand (rows of 64 bf16 along K): lbo unused, sbo = byte step
//     between consecutive 8-row groups; advancing K by 16 elements adds 32 B
//     to the start address.
//   MN-major operand (rows of 64 bf16 along M/N, one row per K index): lbo =
//     byte step between consecutive 64-element M/N chunks, sbo = byte step
//     between consecutive groups of 8 K-rows.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version of the 5th-generation tensor core
  d |= (uint64_t)2 << 61;   // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator; M in {64, 128} (one CTA) or 256 (a CTA pair), N a multiple
// of 16 up to 256.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4)                                  // accumulator format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)           // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | ((uint32_t)(N >> 3) << 17)               // N / 8
         | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// ---------------------------------------------------------------------------
// Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) and Box-Muller
// ---------------------------------------------------------------------------

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
  const uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  const uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t lo0 = kM0 * c.x, hi0 = __umulhi(kM0, c.x);
    const uint32_t lo1 = kM1 * c.z, hi1 = __umulhi(kM1, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// Four standard normals of Philox block `blk` of stream `stream`.
__device__ __forceinline__ void philox_normal4(uint64_t seed, uint32_t stream, uint64_t offset,
                                               uint32_t blk, float (&z)[4]) {
  const U4 x = philox4x32_10(U4{blk, stream, (uint32_t)offset, (uint32_t)(offset >> 32)},
                             (uint32_t)seed, (uint32_t)(seed >> 32));
  const float s24 = 5.9604644775390625e-08f;  // 2^-24
  const float u0 = (float)((x.x >> 8) + 1u) * s24;
  const float v1 = (float)(x.y >> 8) * s24;
  const float u2 = (float)((x.z >> 8) + 1u) * s24;
  const float v3 = (float)(x.w >> 8) * s24;
  const float r0 = sqrtf(-2.0f * logf(u0));
  const float r2 = sqrtf(-2.0f * logf(u2));
  float s, c;
  sincospif(2.0f * v1, &s, &c);
  z[0] = r0 * c;
  z[1] = r0 * s;
  sincospif(2.0f * v3, &s, &c);
  z[2] = r2 * c;
  z[3] = r2 * s;
}

// -2 ln u for u = m 2^-24 (m = 1 .. 2^24), from the SFU's approximate log2.
// That log2 is accurate to an absolute, not a relative, bound, and near
// u = 1 the square root of Box-Muller would magnify the difference (the
// radius sqrt(-2 ln u) is then small).  There, for w = 1 - u <= 1/16 (exact:
// (2^24 - m) 2^-24), the Taylor series -ln(1 - w) = w + w^2/2 + ... + w^6/6
// is used, whose first omitted term is below 2^-24 of the sum.
__device__ __forceinline__ float neg2_log_u(uint32_t m) {
  const float s24 = 5.9604644775390625e-08f;  // 2^-24
  const float u = (float)m * s24;
  const float w = (float)(16777216u - m) * s24;
  float t = fmaf(w, 1.f / 6.f, 0.2f);
  t = fmaf(w, t, 0.25f);
  t = fmaf(w, t, 1.f / 3.f);
  t = fmaf(w, t, 0.5f);
  t = fmaf(w, t, 1.f);
  const float series = 2.f * (w * t);
  return w <= 0.0625f ? series : -2.0f * __logf(u);
}

// The same four normals with the SFU's approximate log2, sine and cosine
// (absolute error of each value below 2e-6 over a 2048 x 8192 draw, against
// the fp64 transform): the Gaussian mechanism's noise,
// drawn by the million inside the gradient kernels, where the full-precision
// transcendentals would cost as many issue slots as the rest of the epilogue.
// The angle 2 pi v is taken as pi + 2 pi (v - 1/2) (v - 1/2 is exact), so the
// SFU sees arguments in [-pi, pi), the range of its stated accuracy, and
// cos and sin change sign.  Probes, whose bf16 rounding is compared exactly,
// keep philox_normal4.
__device__ __forceinline__ void philox_normal4_fast(uint64_t seed, uint32_t stream,
                                                    uint64_t offset, uint32_t blk,
                                                    float (&z)[4]) {
  const U4 x = philox4x32_10(U4{blk, stream, (uint32_t)offset, (uint32_t)(offset >> 32)},
                             (uint32_t)seed, (uint32_t)(seed >> 32));
  const float s24 = 5.9604644775390625e-08f;  // 2^-24
  const float two_pi = 6.28318530717958647692f;
  const float h1 = (float)(x.y >> 8) * s24 - 0.5f;
  const float h3 = (float)(x.w >> 8) * s24 - 0.5f;
  const float r0 = sqrtf(neg2_log_u((x.x >> 8) + 1u));
  const float r2 = sqrtf(neg2_log_u((x.z >> 8) + 1u));
  float s, c;
  __sincosf(two_pi * h1, &s, &c);
  z[0] = -r0 * c;
  z[1] = -r0 * s;
  __sincosf(two_pi * h3, &s, &c);
  z[2] = -r2 * c;
  z[3] = -r2 * s;
}

// Normal number `e` of a stream (used where elements are not block aligned).
__device__ __forceinline__ float philox_normal_at(uint64_t seed, uint32_t stream, uint64_t offset,
                                                  uint64_t e) {
  float z[4];
  philox_normal4(seed, stream, offset, (uint32_t)(e >> 2), z);
  const int lane = (int)(e & 3);
  return lane == 0 ? z[0] : lane == 1 ? z[1] : lane == 2 ? z[2] : z[3];
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): about 16 significant
// bits, so a skinny fp32 operand can enter bf16 MMAs as two products.
__device__ __forceinline__ void split_hilo(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-sample sums of partials, by threads tid = 0 .. nthr-1 of one CTA (all
// of them call it; sync() is a barrier over exactly those threads):
//   sq[i] = scale * sum_{e < count(i)} *ptr(i, e)   (or sq[i] += ..., accumulate)
// Up to kSumSamples samples at once and kSumBatch elements per thread, so a
// thread has kSumSamples * kSumBatch loads in flight: the former sample-by-
// sample loop, two CTA barriers per sample, took ~7 us at the end of the
// persistent GEMMs (per timestamps).  The summation order is fixed (thread
// partition, batch order, shuffle tree, warps in order), so results do not
// depend on timing.  red_smem holds kSumSamples * (nthr / 32) floats; nthr
// is a multiple of 32 and tid / 32 a warp index.
constexpr int kSumSamples = 4;
constexpr int kSumBatch = 8;
template <class Count, class Ptr, class Sync>
__device__ __forceinline__ void sum_per_sample(int B, Count count, Ptr ptr, float scale, float* sq,
                                               bool accumulate, float* red_smem, int tid, int nthr,
                                               Sync sync) {
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = nthr >> 5;
  for (int i0 = 0; i0 < B; i0 += kSumSamples) {
    long long cnt[kSumSamples];
    long long nmax = 0;
#pragma unroll
    for (int j = 0; j < kSumSamples; ++j) {
      cnt[j] = i0 + j < B ? count(i0 + j) : 0;
      nmax = cnt[j] > nmax ? cnt[j] : nmax;
    }
    float acc[kSumSamples];
#pragma unroll
    for (int j = 0; j < kSumSamples; ++j) acc[j] = 0.f;
    for (long long e0 = tid; e0 < nmax; e0 += (long long)kSumBatch * nthr) {
      float v[kSumSamples][kSumBatch];
#pragma unroll
      for (int j = 0; j < kSumSamples; ++j)
#pragma unroll
        for (int q = 0; q < kSumBatch; ++q) {
          const long long e = e0 + (long long)q * nthr;
          v[j][q] = e < cnt[j] ? __ldcg(ptr(i0 + j, e)) : 0.f;
        }
#pragma unroll
      for (int j = 0; j < kSumSamples; ++j)
#pragma unroll
        for (int q = 0; q < kSumBatch; ++q) acc[j] += v[j][q];
    }
#pragma unroll
    for (int j = 0; j < kSumSamples; ++j) {
      const float a = warp_sum(acc[j]);
      if (lane == 0) red_smem[j * nwarps + warp] = a;
    }
    sync();
    if (tid < kSumSamples && i0 + tid < B) {
      const int i = i0 + tid;
      float s = 0.f;
      for (int w = 0; w < nwarps; ++w) s += red_smem[tid * nwarps + w];
      sq[i] = accumulate ? sq[i] + scale * s : scale * s;
    }
    sync();
  }
}

// The last CTA to finish a kernel (integer ticket) computes
//   sq[i] = scale * sum_{u < nunits, w < nw} part[(u*su + i*si)*nw + w].
// Every thread of every CTA calls it once at the end of the kernel, one
// sample after the other with few registers (kernels whose producer warps
// have given theirs away call it).  The summation order is fixed (thread
// partition, 8-wide batches, shuffle tree, warps in order), so results do not
// depend on CTA timing.  `ticket` must be zero at launch; the last CTA resets
// it.  With `accumulate`, sq[i] += the result instead.
__device__ __forceinline__ void reduce_partials_last_cta(const float* part, int B, int nunits,
                                                         long long su, long long si, int nw,
                                                         float scale, float* sq,
                                                         uint32_t* ticket, float* red_smem,
                                                         int* flag_smem, bool accumulate = false) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *flag_smem = (atomicAdd(ticket, 1u) == gridDim.x - 1u) ? 1 : 0;
  __syncthreads();
  if (!*flag_smem) return;
  __threadfence();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (int)(blockDim.x >> 5);
  const long long n = (long long)nunits * nw;
  for (int i = 0; i < B; ++i) {
    float acc = 0.f;
    for (long long e0 = threadIdx.x; e0 < n; e0 += 8ll * blockDim.x) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const long long e = e0 + (long long)q * blockDim.x;
        v[q] = e < n ? __ldcg(part + ((e / nw) * su + (long long)i * si) * nw + (e % nw)) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) acc += v[q];
    }
    acc = warp_sum(acc);
    if (lane == 0) red_smem[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < nwarps; ++w) s += red_smem[w];
      sq[i] = accumulate ? sq[i] + scale * s : scale * s;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *ticket = 0u;
}

// FIBER step of one parameter element ("Technical summary: FIBER", Method A
// and C): the innovation filter on g = grad * inv_denom, then AdamW on the
// filtered gradient with the second moment reduced by A(omega) s2.
__device__ __forceinline__ void fiber_elem(const FiberDev& f, float grad, float& theta, float& gf,
                                           float& r, float& m, float& v) {
  const float g = grad * f.inv_denom;
  r = fmaf(f.omega, g - gf, (1.f - f.omega) * r);
  gf += r;
  m = fmaf(f.beta1, m, (1.f - f.beta1) * gf);
  v = fmaf(f.beta2, v, (1.f - f.beta2) * gf * gf);
  const float vbar = fmaxf(v * f.bc2 - f.calib, f.eps_v);
  theta -= f.lr * ((m * f.bc1) / (sqrtf(vbar) + f.eps) + f.wd * theta);
}

// The same on four consecutive elements e .. e + 3 (16-byte aligned).
__device__ __forceinline__ void fiber_update4(const FiberDev& f, size_t e, float4 g) {
  float4 th = *reinterpret_cast<const float4*>(f.param + e);
  float4 gf = *reinterpret_cast<const float4*>(f.filt + e);
  float4 r = *reinterpret_cast<const float4*>(f.resid + e);
  float4 m = *reinterpret_cast<const float4*>(f.m + e);
  float4 v = *reinterpret_cast<const float4*>(f.v + e);
  fiber_elem(f, g.x, th.x, gf.x, r.x, m.x, v.x);
  fiber_elem(f, g.y, th.y, gf.y, r.y, m.y, v.y);
  fiber_elem(f, g.z, th.z, gf.z, r.z, m.z, v.z);
  fiber_elem(f, g.w, th.w, gf.w, r.w, m.w, v.w);
  *reinterpret_cast<float4*>(f.param + e) = th;
  *reinterpret_cast<float4*>(f.filt + e) = gf;
  *reinterpret_cast<float4*>(f.resid + e) = r;
  *reinterpret_cast<float4*>(f.m + e) = m;
  *reinterpret_cast<float4*>(f.v + e) = v;
}

__device__ __forceinline__ void fiber_update1(const FiberDev& f, size_t e, float g) {
  fiber_elem(f, g, f.param[e], f.filt[e], f.resid[e], f.m[e], f.v[e]);
}

}  // namespace dpclip
