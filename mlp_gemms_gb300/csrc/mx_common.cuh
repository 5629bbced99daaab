// Device-side building blocks shared by the MX kernels (sm_103a).
//
// * Exact round-up (RCEIL) E8M0 block scales from the fp32 bit fields, and
//   the element packers built on the hardware's saturating round-to-nearest
//   conversions (cvt.rn.satfinite.{e4m3,e2m3,e2m1}x2.f32).
//   torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
//   group gemm", correctness-first kernels commit: E8M0 rounds upward, the
//   f32->E4M3 conversion equals torch's cast, amax propagates NaN.
// * Thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk[.tensor]) and
//   the 5th-generation tensor core (tcgen05.{alloc,cp,mma,commit,ld}).
// * Bounded waits: every spin on an mbarrier gives up after a time budget,
//   records MX device status "timeout" and lets the kernel unwind.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mx {

enum Fmt : int { E4M3 = 0, E2M3 = 1, E2M1 = 2 };

// Device status words (one set per translation unit that includes this).
// bit 0: a bounded wait ran out; bit 1: malformed offsets seen on device;
// bit 2: a routing index (expert id or source row) out of range.
enum : unsigned { DEV_TIMEOUT = 1u, DEV_BAD_OFFSETS = 2u, DEV_BAD_INDEX = 4u };
// Longest any bounded device-side wait spins before it gives up.
constexpr uint64_t WAIT_BUDGET_NS = 2000000000ull;

// ---------------------------------------------------------------------------
// Element formats
// ---------------------------------------------------------------------------

// Largest finite value emax = 1.m_x * 2^E_x of each element format, as the
// unbiased exponent and the 23-bit fp32 mantissa field of 1.m_x.
template <int FMT> struct FmtMax;
template <> struct FmtMax<E4M3> { static constexpr int E = 8; static constexpr uint32_t M = 0x600000u; };  // 448 = 1.75*2^8
template <> struct FmtMax<E2M3> { static constexpr int E = 2; static constexpr uint32_t M = 0x700000u; };  // 7.5 = 1.875*2^2
template <> struct FmtMax<E2M1> { static constexpr int E = 2; static constexpr uint32_t M = 0x400000u; };  // 6 = 1.5*2^2

// Block scale byte from the NaN-propagating amax given as fp32 bits of |x|
// (a larger-than-Inf pattern means a NaN was seen).  The scale is the
// smallest e with amax <= emax * 2^e: with amax = 1.m_a * 2^E_a this is
// E_a - E_x + (m_a > m_x), clamped to [-127, 127].
template <int FMT>
__device__ __forceinline__ uint32_t rceil_scale_byte(uint32_t amax_bits) {
  if (amax_bits > 0x7F800000u) return 0xFFu;   // NaN
  if (amax_bits == 0x7F800000u) return 0xFEu;  // +Inf
  if (amax_bits == 0u) return 0u;
  int E;
  uint32_t m;
  if ((amax_bits >> 23) == 0u) {               // fp32 subnormal: normalise
    int lz = __clz(amax_bits) - 8;
    m = (amax_bits << lz) & 0x7FFFFFu;
    E = -118 - __clz(amax_bits);
  } else {
    E = (int)(amax_bits >> 23) - 127;
    m = amax_bits & 0x7FFFFFu;
  }
  int e = E - FmtMax<FMT>::E + (m > FmtMax<FMT>::M ? 1 : 0);
  e = e < -127 ? -127 : (e > 127 ? 127 : e);
  return (uint32_t)(e + 127);
}

// The same byte as rceil_scale_byte: as a biased byte the scale is the
// biased exponent field minus E_x plus the carry, clamped to [0, 254].
// Zero and fp32 subnormals land below 0 for every format here (E_x >= 2),
// so the clamp gives them byte 0; +Inf gives 0xFE and NaN 0xFF.  Written
// without branches (selects only).  Measured on GB300: faster in the GEMM
// epilogues, which interleave many independent blocks per thread; slower
// in the quantizer kernel, which keeps rceil_scale_byte.
template <int FMT>
__device__ __forceinline__ uint32_t rceil_scale_byte_sel(uint32_t amax_bits) {
  static_assert(FmtMax<FMT>::E >= 2, "zero/subnormal amax must clamp to byte 0");
  int b = (int)(amax_bits >> 23) - FmtMax<FMT>::E + ((amax_bits & 0x7FFFFFu) > FmtMax<FMT>::M ? 1 : 0);
  b = b < 0 ? 0 : (b > 254 ? 254 : b);
  const uint32_t special = amax_bits == 0x7F800000u ? 0xFEu : 0xFFu;
  return amax_bits >= 0x7F800000u ? special : (uint32_t)b;
}

// 2^-(b-127) as an fp32 multiplier for scale byte b in [0, 254].
__device__ __forceinline__ float inv_scale_from_byte(uint32_t b) {
  int neg_e = 127 - (int)b;                    // -e in [-127, 127]
  uint32_t bits = neg_e >= -126 ? (uint32_t)(neg_e + 127) << 23 : 0x00400000u;  // 2^-127 is subnormal
  return __uint_as_float(bits);
}

// Two fp32 values -> two codes; lo lands in the low byte / nibble.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e2m3x2(float lo, float hi) {
  uint16_t r;  // each 6-bit code in the low bits of its byte
  asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Bytes of packed payload for one block of 32 elements.
template <int FMT> struct BlockBytes;
template <> struct BlockBytes<E4M3> { static constexpr int value = 32; };
template <> struct BlockBytes<E2M3> { static constexpr int value = 24; };
template <> struct BlockBytes<E2M1> { static constexpr int value = 16; };

// Quantize 32 fp32 values (already scaled by 2^-e, or NaN block) into the
// packed payload words of one block: E4M3 8 words, E2M3 6 words (four 6-bit
// codes per 24 bits, little-endian bit stream), E2M1 4 words (even element
// in the low nibble).
template <int FMT>
__device__ __forceinline__ void pack_block(const float (&v)[32], uint32_t (&w)[8]) {
  if constexpr (FMT == E4M3) {
#pragma unroll
    for (int i = 0; i < 8; i++)
      w[i] = cvt_e4m3x2(v[4 * i], v[4 * i + 1]) | (cvt_e4m3x2(v[4 * i + 2], v[4 * i + 3]) << 16);
  } else if constexpr (FMT == E2M1) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      uint32_t b0 = cvt_e2m1x2(v[8 * i + 0], v[8 * i + 1]);
      uint32_t b1 = cvt_e2m1x2(v[8 * i + 2], v[8 * i + 3]);
      uint32_t b2 = cvt_e2m1x2(v[8 * i + 4], v[8 * i + 5]);
      uint32_t b3 = cvt_e2m1x2(v[8 * i + 6], v[8 * i + 7]);
      w[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
  } else {
    // 8 groups of 4 codes -> 24 bits each; 32 codes -> 24 bytes = 6 words.
    uint32_t g[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      uint32_t p0 = cvt_e2m3x2(v[4 * i], v[4 * i + 1]);
      uint32_t p1 = cvt_e2m3x2(v[4 * i + 2], v[4 * i + 3]);
      uint32_t c0 = p0 & 0x3Fu, c1 = (p0 >> 8) & 0x3Fu, c2 = p1 & 0x3Fu, c3 = (p1 >> 8) & 0x3Fu;
      g[i] = c0 | (c1 << 6) | (c2 << 12) | (c3 << 18);
    }
#pragma unroll
    for (int j = 0; j < 2; j++) {  // 4 groups (96 bits) -> 3 words
      uint32_t a = g[4 * j], b = g[4 * j + 1], c = g[4 * j + 2], d = g[4 * j + 3];
      w[3 * j + 0] = a | (b << 24);
      w[3 * j + 1] = (b >> 8) | (c << 16);
      w[3 * j + 2] = (c >> 16) | (d << 8);
    }
  }
}

// NaN block: every element code is the format's NaN (E4M3) or +0.
template <int FMT>
__device__ __forceinline__ uint32_t nan_block_word() { return FMT == E4M3 ? 0x7F7F7F7Fu : 0u; }

// max(|a|, |b|) in magnitude (the sign bit is meaningless), NaN if either is.
__device__ __forceinline__ float max_abs_nan(float a, float b) {
  float d;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// fp32 bits of max |v[i]| over N values (a power of two), by a pairwise tree;
// any NaN gives a larger-than-Inf pattern, as rceil_scale_byte expects.
template <int N>
__device__ __forceinline__ uint32_t amax_abs_bits(const float* v) {
  float t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; i++) t[i] = max_abs_nan(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int w = N / 4; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; i++) t[i] = max_abs_nan(t[i], t[i + w]);
  }
  return __float_as_uint(t[0]) & 0x7FFFFFFFu;
}

// v[i] *= s for N (even) values, two lanes per instruction (each lane an
// ordinary round-to-nearest fp32 product).
template <int N>
__device__ __forceinline__ void scale_values(float* v, float s) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    uint64_t p, q;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(v[i]), "f"(v[i + 1]));
    asm("mov.b64 %0, {%1, %1};" : "=l"(q) : "f"(s));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(p) : "l"(q));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v[i]), "=f"(v[i + 1]) : "l"(p));
  }
}

// Scale (by 2^-e) and pack one block whose scale byte is `sb`.
template <int FMT>
__device__ __forceinline__ void quantize_block_words(float (&v)[32], uint32_t sb, uint32_t (&w)[8]) {
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; i++) w[i] = nan_block_word<FMT>();
    return;
  }
  scale_values<32>(v, inv_scale_from_byte(sb));
  pack_block<FMT>(v, w);
}

// (a0, a1), (b0, b1) -> (a0 + b0, a1 + b1), (a0 - b0, a1 - b1): two
// butterflies in one packed add and one packed subtract (each lane an
// ordinary round-to-nearest fp32 operation).
__device__ __forceinline__ void butterfly_pair(float& a0, float& a1, float& b0, float& b1) {
  uint64_t A, B, S, D;
  asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b0), "f"(b1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(S) : "l"(A), "l"(B));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(D) : "l"(A), "l"(B));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(S));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(D));
}

// In-place butterfly stages of stride 1, 2, ..., N/2 over N values
// (v[i], v[i+h]) -> (v[i] + v[i+h], v[i] - v[i+h]); stride 1 scalar, the
// wider strides two butterflies at a time.
template <int N>
__device__ __forceinline__ void butterfly_stages(float* v) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = __fadd_rn(a, b);
    v[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      if (i & h) continue;
      butterfly_pair(v[i], v[i + 1], v[i + h], v[i + h + 1]);
    }
  }
}

// In-register 32-point Hadamard: five butterfly stages (stride 1..16), then
// one multiply by fl32(1/sqrt(32)).  Primus PR #1064 "feat(mxfp6): MXFP6
// (E2M3) Flux linears, a fused MLP, and the MLPerf recipe", first commit:
// the rotation folded into the packer.
__device__ __forceinline__ void hadamard32(float (&v)[32]) {
  butterfly_stages<32>(v);
  scale_values<32>(v, __uint_as_float(0x3E3504F3u));  // fl32(1/sqrt(32))
}

// Offset of scale (r, c) in the blocked layout of a [rows, scale_cols] scale
// matrix (128-row x 4-column chunks of 512 bytes, padding zero).
__host__ __device__ __forceinline__ int64_t blocked_offset(int64_t r, int64_t c, int64_t scale_cols) {
  int64_t cpad4 = (scale_cols + 3) / 4;
  return ((r >> 7) * cpad4 + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// ---------------------------------------------------------------------------
// Bounded waits and shared-memory / TMA / mbarrier primitives
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up when the
// CTA-wide abort flag is raised or after `budget_ns`; returns false then.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > budget_ns) { *abort_flag = 1; return false; }
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load of box (c0 innermost, c1) into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(cache_hint)
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// 2-D tiled TMA store of a shared-memory box to global memory (bulk group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               :: "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(src)) : "memory");
}
// 2-D tiled TMA reduce-add of a shared-memory box into global memory
// (element type from the tensor map; one rounding per element).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];"
               :: "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(src)) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory sources of all committed bulk stores have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// All committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(map) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (tensor memory + 5th-gen MMA)
// ---------------------------------------------------------------------------

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(slot)), "n"(NCOLS) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "n"(NCOLS) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), fixed version bits 46..47 = 1, layout
// type in bits 61..63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// Copy one 512-byte blocked scale chunk (32 rows x 128 bits, replicated to
// the four 32-lane quarters) from shared memory into tensor memory.
__device__ __forceinline__ void tc_copy_scales(uint32_t taddr, uint32_t saddr) {
  uint64_t d = smem_desc(saddr, 0, 128, 0);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(d) : "memory");
}

// Instruction descriptor of tcgen05.mma .kind::mxf8f6f4.block_scale with
// fp32 accumulation, K-major A and B, UE8M0 scales.
__host__ __device__ constexpr uint32_t mma_idesc_mx(uint32_t atype, uint32_t btype, uint32_t M, uint32_t N,
                                                    uint32_t a_sf_id, uint32_t b_sf_id) {
  return (b_sf_id << 4) | (atype << 7) | (btype << 10) | ((N >> 3) << 17) | (1u << 23) |
         ((M >> 4) << 24) | (a_sf_id << 29);
}

// D[tmem] (+)= (A * 2^sfa) (B * 2^sfb)^T for one K=32 step.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Element type code of E2M1 in the .kind::mxf4 instruction descriptor.
constexpr uint32_t MXF4_E2M1 = 1;

// D[tmem] (+)= (A * 2^sfa) (B * 2^sfb)^T for one K=64 step of packed E2M1
// operands (two elements per byte, 32 bytes of each row), two scale bytes
// per row: scale IDs 0 and 2 pick the first or second pair of the four
// bytes a tensor-memory scale word holds.
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The warp's 32 lanes x 32 consecutive columns of tensor memory from 32
// registers per thread (the mirror of tmem_ld32); complete once
// tmem_wait_st() returns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
         "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
         "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier among `nthreads` threads (id 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t elect_one_lane() {
  uint32_t pred;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// fp32 -> bf16 bits, round to nearest even (hardware conversion).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace mx
