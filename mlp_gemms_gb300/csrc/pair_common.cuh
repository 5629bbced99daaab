// Primitives for CTA pairs (clusters of two CTAs sharing tcgen05
// .cta_group::2 MMAs): cluster rank and addressing, cluster-scope waits and
// arrivals, 2-SM TMA loads whose bytes complete on the leader CTA's barrier,
// the pair forms of the scale copy, MMA and commit, and the table of 256-row
// tiles per expert segment.  Used by the plain pair GEMM (gemm_pair.cu) and
// by the pair instantiations of the fused-epilogue kernel (gemm_kernel.cuh).
#pragma once
#include "mx_common.cuh"

namespace mx {

constexpr int MAX_PAIR_G = 1024;  // experts the row-tile table holds

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The leader CTA's (rank 0) shared::cluster address of a local shared address.
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bounded wait with cluster-scope acquire (the barrier's arrivals come from
// both CTAs of the pair).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
    if ((++n & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > WAIT_BUDGET_NS) { *abort_flag = 1; return false; }
    }
  }
}
// The peer CTA's (rank 1) shared::cluster address of a local shared address.
__device__ __forceinline__ uint32_t peer_addr(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 1;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
// A 32-bit store into the shared memory of a CTA of the cluster.
__device__ __forceinline__ void st_cluster_u32(uint32_t addr_cl, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr_cl), "r"(v) : "memory");
}
__device__ __forceinline__ void arrive_on_leader(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar_cl) : "memory");
}
// 2-SM TMA loads: destination in this CTA's shared memory, completion bytes
// counted on the (leader's) barrier at shared::cluster address bar_cl.
__device__ __forceinline__ void tma2_load_2d(void* dst, const CUtensorMap* m, int c0, int c1, uint32_t bar_cl,
                                             uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
               " [%0], [%1, {%2, %3}], [%4], %5;"
               :: "r"(smem_u32(dst)), "l"(m), "r"(c0), "r"(c1), "r"(bar_cl), "l"(pol) : "memory");
}
__device__ __forceinline__ void tma2_load_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint32_t bar_cl) {
  asm volatile("cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_u32(dst)), "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cl) : "memory");
}
__device__ __forceinline__ void tc2_copy_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc2_mma_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
__device__ __forceinline__ void tc2_mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                             uint32_t sfb, uint32_t accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
// Arrive on the barrier at this shared offset in both CTAs once every
// tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void tc2_commit_both(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(smem_u32(bar)), "h"((uint16_t)3) : "memory");
}
__device__ __forceinline__ void tc2_commit_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}


// Row tiles of 256 per expert segment (segments are multiples of 128 rows;
// an odd number of 128-row blocks leaves the last tile's upper half past the
// segment: computed, not stored).  pref[g] = row tiles of experts 0..g-1,
// built in shared memory by one warp with a running warp scan; a malformed
// segment (not a multiple of 128 rows, decreasing, or past R) gets no tiles
// and sets the malformed-offsets bit in *status when status is not null.
__device__ __forceinline__ void build_pair_prefix(const int32_t* offsets, int G, int64_t R, int32_t* pref, int lane,
                                                  unsigned* status) {
  int32_t run = 0;
  if (lane == 0) pref[0] = 0;
  bool bad = false;
  for (int base = 0; base < G; base += 32) {
    const int g = base + lane;
    int32_t cnt = 0;
    if (g < G) {
      const int64_t end = offsets ? (int64_t)__ldg(offsets + g) : R;
      const int64_t start = (offsets && g) ? (int64_t)__ldg(offsets + g - 1) : 0;
      if ((start & 127) || (end & 127) || end < start || end > R) bad = true;
      else cnt = (int32_t)((end - start + 255) / 256);
    }
    int32_t v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (g < G) pref[g + 1] = run + v;
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  if (status != nullptr && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, DEV_BAD_OFFSETS);
}

// Row tile mt (in expert order) -> its expert g, row base m0 and whether its
// upper 128 rows lie inside the segment; false when mt is past the last tile.
__device__ __forceinline__ bool pair_row_tile(const int32_t* offsets, int G, int64_t R, const int32_t* pref,
                                              int64_t mt, int* g_out, int64_t* m0_out, int* upper_out) {
  if (mt >= pref[G]) return false;
  int lo = 0, hi = G - 1;  // the expert g with pref[g] <= mt < pref[g + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)pref[mid] <= mt) lo = mid; else hi = mid - 1;
  }
  const int64_t start = (offsets && lo) ? (int64_t)__ldg(offsets + lo - 1) : 0;
  const int64_t end = offsets ? (int64_t)__ldg(offsets + lo) : R;
  *g_out = lo;
  *m0_out = start + 256 * (mt - pref[lo]);
  *upper_out = *m0_out + 128 < end ? 1 : 0;
  return true;
}

}  // namespace mx
