// The grouped block-scaled GEMM on CTA pairs (tcgen05 .cta_group::2), BF16
// out: y[r, :] = A[r, :] B[g]^T for the rows r of expert g's segment.
//
// torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
// group gemm", cudnn-fe ops commit: its kernels take 256-row MMA tiles on
// two SMs and need every expert's segment to be a multiple of 256 rows.
// This one takes 128-row segments too: an expert with an odd number of
// 128-row blocks computes its last tile's upper half and does not store it.
//
// A pair of CTAs (a cluster of two) takes a 256 x 256 output tile: each CTA
// loads its own 128 rows of A and its own half (128 rows) of the tile's B
// slice, plus the scale chunks of its A rows and of all 256 B rows, by 2-SM
// TMA loads whose bytes are all counted on the leader CTA's stage barrier.
// The leader's MMA thread issues tcgen05.mma .cta_group::2 (M = 256, N = 256,
// K = 32 on .kind::mxf8f6f4; K = 64 on .kind::mxf4 for packed E2M1 operands,
// whose stages hold 256 K-elements and two scale chunks), each CTA's tensor
// memory holding its 128 x 256 fp32 accumulator,
// and its commits arrive on both CTAs' barriers.  A warp of the leader of
// its own copies each stage's scale chunks into both CTAs' tensor memory
// (tcgen05.cp .cta_group::2) and signals the MMA thread, which then issues
// only MMAs (with the copies inline the issuing thread, feeding two SMs'
// tensor cores, was the limit).  Each CTA's eight epilogue
// warps read their accumulator, hand it back to the leader (the peer's by
// one remote arrive on the leader's barrier) and store BF16 by TMA.  Tensor memory is
// allocated by both CTAs collectively (.cta_group::2 returns the same
// columns in both, checked on the device before this kernel was written).
// Every wait is bounded; on expiry the CTA records a device status bit and
// unwinds.  No TMA multicast.
#include "gemm_kernel.cuh"

namespace mx {

static __device__ unsigned g_pair_status = 0;

namespace pair {
constexpr int THREADS = 352;                          // producer, MMA, 8 epilogue warps, scale copies
constexpr int SCALE_WARP = 10;
constexpr uint32_t SF_TMEM = 256;                     // scale slots after the accumulator
// F4: packed E2M1 operands on .kind::mxf4 -- a stage's 128-byte rows hold
// 256 K-elements, i.e. KC = 2 scale chunks per 128-row block.
template <bool F4> struct PCfg {
  static constexpr int KC = F4 ? 2 : 1;
  static constexpr int ST = F4 ? 5 : 6;               // 33.5 KB (35 KB with F4) stages
  static constexpr int A_BYTES = 16384, B_BYTES = 16384;
  // A's KC chunks, then B's two row blocks of KC chunks each
  static constexpr int SF_BYTES = KC * 1536;
  static constexpr int SF_COLS = KC * 12;             // tensor-memory columns of a stage's scales
  static constexpr int OFF_B = ST * A_BYTES;
  static constexpr int OFF_SF = OFF_B + ST * B_BYTES;
  static constexpr int OFF_BAR = OFF_SF + ST * SF_BYTES;
  // full, empty, acc_full, acc_empty, final, peer_read, sf_ready[ST], sf_final
  static constexpr int NUM_BARS = 3 * ST + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem slot, abort flag
  static constexpr int OFF_STG = (OFF_MISC + 64 + 1023) / 1024 * 1024;  // eight 2 KB staging buffers
  static constexpr int OFF_PREF = OFF_STG + 8 * 2048;     // pair row tiles before expert g, g = 0..G
  static constexpr int SMEM = OFF_PREF + 4 * (MAX_PAIR_G + 1) + 1024;  // + slack for 1024-byte alignment
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(SF_TMEM + ST * SF_COLS <= 512, "scale slots must fit");
};
}  // namespace pair

struct PairTile {
  int active, g;
  int64_t m0, n0;
  int upper;  // the tile's rows m0 + 128 .. m0 + 255 belong to its expert
};

// Pair tile t -> (expert, row base of its 256-row tile, column base): row
// tile mt = t / n_tiles in expert order (pref), column tile t % n_tiles.
__device__ __forceinline__ PairTile get_pair_tile(const PairParams& p, const int32_t* pref, int64_t t) {
  PairTile T;
  T.active = 0; T.g = 0; T.upper = 0; T.m0 = 0;
  T.n0 = (t % p.n_tiles) * 256;
  T.active = pair_row_tile(p.offsets, p.G, p.R, pref, t / p.n_tiles, &T.g, &T.m0, &T.upper) ? 1 : 0;
  return T;
}

template <bool F4>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::THREADS, 1)
mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                    const __grid_constant__ CUtensorMap tmO, const PairParams p) {
  using namespace pair;
  using C = PCfg<F4>;
  constexpr int ST = C::ST, KC = C::KC;
  constexpr int A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, SF_BYTES = C::SF_BYTES;
  constexpr int OFF_B = C::OFF_B, OFF_SF = C::OFF_SF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);  // leader's: both CTAs' bytes of a stage
  uint64_t* empty = full + ST;                                   // both CTAs: the stage's MMAs are done
  uint64_t* acc_full = empty + ST;                               // both CTAs: the tile's MMAs are done
  uint64_t* acc_empty = acc_full + 1;   // leader's: its 8 epilogue warps and the peer's hand-off have read
  uint64_t* final_bar = acc_empty + 1;
  uint64_t* peer_read = final_bar + 1;  // peer's: its 8 epilogue warps have read their accumulator
  uint64_t* sf_ready = peer_read + 1;   // leader's: the stage's scales are in both CTAs' tensor memory
  uint64_t* sf_final = sf_ready + ST;   // leader's: every scale copy has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 9);
    mbar_init(final_bar, 1);
    mbar_init(peer_read, 8);
    for (int s2 = 0; s2 < ST; s2++) mbar_init(&sf_ready[s2], 1);
    mbar_init(sf_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA); prefetch_tensormap(&tmB); prefetch_tensormap(&tmSA); prefetch_tensormap(&tmSB);
    prefetch_tensormap(&tmO);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  int32_t* pref = reinterpret_cast<int32_t*>(smem + C::OFF_PREF);
  if (warp == 0) build_pair_prefix(p.offsets, p.G, p.R, pref, lane, leader ? &g_pair_status : nullptr);
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive or copy; pref is built
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int64_t pidx = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int nc = (int)(p.K / 128);        // 128-K scale chunks
  const int nk = (nc + KC - 1) / KC;     // stages per tile

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_normal(), pol_b = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int armed[ST];
      for (int s = 0; s < ST; s++) armed[s] = -1;
      bool ok = true;
      for (int64_t t = pidx; t < p.num_tiles && ok; t += npairs) {
        const PairTile T = get_pair_tile(p, pref, t);
        if (!T.active) continue;
        const int64_t brow = (int64_t)T.g * p.Nb + T.n0;
        for (int kb = 0; kb < nk; kb++) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          const uint32_t fb = leader_addr(&full[stage]);
          if (leader) {
            mbar_arrive_expect_tx(&full[stage], 2u * p.tx_bytes);
            armed[stage] = (int)phase;
          }
          // x: 128 elements (F4: 128 bytes = 256 packed elements) per stage.
          // F4's last stage of an odd chunk count reads its second half past
          // K: zero-filled and counted like the rest of the box, read by no MMA.
          tma2_load_2d(smem + stage * A_BYTES, &tmA, kb * 128, (int)(T.m0 + 128 * rank), fb, pol_a);
          tma2_load_2d(smem + OFF_B + stage * B_BYTES, &tmB, kb * 128, (int)(brow + 128 * rank), fb, pol_b);
          uint8_t* sf = smem + OFF_SF + stage * SF_BYTES;
          tma2_load_3d(sf, &tmSA, 0, kb * KC, (int)((T.m0 >> 7) + rank), fb);
          tma2_load_3d(sf + KC * 512, &tmSB, 0, kb * KC, (int)(brow >> 7), fb);
          if (++stage == ST) { stage = 0; phase ^= 1u; }
        }
      }
      // The leader's stage barriers count both CTAs' copies: every copy has
      // landed once they complete (the drain ignores the abort flag).
      if (leader) {
        volatile int no_abort = 0;
        for (int s = 0; s < ST; s++)
          if (armed[s] >= 0) mbar_wait_bounded(&full[s], (uint32_t)armed[s], &no_abort, WAIT_BUDGET_NS);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      const uint64_t a_desc0 = smem_desc(smem_u32(smem), 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(smem_u32(smem + OFF_B), 16, 1024, 2);
      const uint32_t idesc0 = F4 ? mma_idesc_mx(MXF4_E2M1, MXF4_E2M1, 256, 256, 0, 0)
                                 : mma_idesc_mx((uint32_t)p.a_type, (uint32_t)p.b_type, 256, 256, 0, 0);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t t = pidx; t < p.num_tiles && ok; t += npairs) {
        const PairTile T = get_pair_tile(p, pref, t);
        if (!T.active) continue;
        if (!mbar_wait_cluster(acc_empty, acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nk; kb++) {
          // the stage's operands have landed and its scales are in tensor memory
          if (!mbar_wait_bounded(&sf_ready[stage], phase, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + SF_TMEM + (uint32_t)(stage * C::SF_COLS);
          const uint64_t ad = a_desc0 + (uint64_t)((stage * A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)((stage * B_BYTES) >> 4);
          if constexpr (F4) {
            const int nch = (2 * kb + 1 < nc) ? 2 : 1;
#pragma unroll
            for (int j = 0; j < 4; j++) {
              if (j < 2 * nch) {  // K = 64 per MMA; scale IDs 0 and 2 pick the chunk's byte pair
                const uint32_t sid = (uint32_t)(j & 1) * 2u;
                tc2_mma_mxf4(tmem_base, ad + 2 * j, bd + 2 * j, idesc0 | (sid << 4) | (sid << 29),
                             sf_t + 4 * (j >> 1), sf_t + 8 + 8 * (j >> 1), (kb | j) != 0 ? 1u : 0u);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; j++)
              tc2_mma_mx(tmem_base, ad + 2 * j, bd + 2 * j, idesc0 | ((uint32_t)j << 4) | ((uint32_t)j << 29), sf_t,
                         sf_t + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc2_commit_both(&empty[stage]);
          if (++stage == ST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc2_commit_both(acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) *abort_flag = 1;
      // No MMA may still be writing either CTA's tensor memory when it is freed.
      volatile int no_abort = 0;
      tc2_commit_local(final_bar);
      mbar_wait_bounded(final_bar, 0, &no_abort, WAIT_BUDGET_NS);
    }
  } else if (warp == SCALE_WARP) {
    // ------------------------------------------------------------ scale copies (leader)
    // In the MMA thread's stage order: wait for the stage's bytes (both
    // CTAs'), copy its scale chunks into both CTAs' tensor memory and signal
    // sf_ready once the copies have completed.  A slot is rewritten only after
    // the producers refilled its stage, i.e. after the MMAs that read it.
    if (lane == 0 && leader) {
      const uint64_t sf_desc0 = smem_desc(smem_u32(smem + OFF_SF), 0, 128, 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t t = pidx; t < p.num_tiles && ok; t += npairs) {
        const PairTile T = get_pair_tile(p, pref, t);
        if (!T.active) continue;
        for (int kb = 0; kb < nk; kb++) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + SF_TMEM + (uint32_t)(stage * C::SF_COLS);
          const uint64_t sd = sf_desc0 + (uint64_t)((stage * SF_BYTES) >> 4);
          if constexpr (F4) {
            // A's chunk c at column 4c (each CTA its own rows), B's chunk c of
            // row block i at 8 + 8c + 4i; shared memory holds A's chunks, then
            // B's row blocks of two chunks
            const int nch = (2 * kb + 1 < nc) ? 2 : 1;
#pragma unroll
            for (int c = 0; c < 2; c++) {
              if (c < nch) {
                tc2_copy_scales(sf_t + 4 * c, sd + (uint64_t)((512 * c) >> 4));
#pragma unroll
                for (int i = 0; i < 2; i++)
                  tc2_copy_scales(sf_t + 8 + 8 * c + 4 * i, sd + (uint64_t)((1024 + 512 * (2 * i + c)) >> 4));
              }
            }
          } else {
            tc2_copy_scales(sf_t, sd);                   // A's 128 rows (each CTA its own)
            tc2_copy_scales(sf_t + 4, sd + (512 >> 4));  // B rows 0..127 of the tile
            tc2_copy_scales(sf_t + 8, sd + (1024 >> 4)); // B rows 128..255
          }
          tc2_commit_local(&sf_ready[stage]);
          if (++stage == ST) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) *abort_flag = 1;
      // No copy may still be writing either CTA's tensor memory when it is freed.
      volatile int no_abort = 0;
      tc2_commit_local(sf_final);
      mbar_wait_bounded(sf_final, 0, &no_abort, WAIT_BUDGET_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;            // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;  // column half of the 256-column tile
    uint8_t* stg = smem + C::OFF_STG + (warp - 2) * 2048;
    const uint32_t acc_empty_cl = leader_addr(acc_empty);
    const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
    uint32_t acc_phase = 0, peer_phase = 0;
    for (int64_t t = pidx; t < p.num_tiles; t += npairs) {
      const PairTile T = get_pair_tile(p, pref, t);
      if (!T.active) continue;
      if (!mbar_wait_bounded(acc_full, acc_phase, abort_flag, WAIT_BUDGET_NS)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; c++) tmem_ld32(tbase + 32 * c, v[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      // Hand the accumulator back: the leader's warps arrive on its barrier
      // directly; the peer's warps meet on their own barrier and one thread
      // then makes a single arrival across the pair (one remote message per
      // tile instead of eight: the hand-back 1.18 -> 0.88 us per tile).
      if (leader) {
        if (lane == 0) mbar_arrive(acc_empty);
      } else {
        if (lane == 0) mbar_arrive(peer_read);
        if (warp == 2) {
          const bool okp = mbar_wait_bounded(peer_read, peer_phase, abort_flag, WAIT_BUDGET_NS);
          peer_phase ^= 1u;
          if (!okp) break;
          if (lane == 0) arrive_on_leader(acc_empty_cl);
        }
      }
      if (p.bias != nullptr) {  // bias added to the fp32 accumulator: one rounding
        const uint4* bp = reinterpret_cast<const uint4*>(p.bias + (int64_t)T.g * p.bias_ld + T.n0 + half * 128);
#pragma unroll
        for (int c = 0; c < 4; c++) {
#pragma unroll
          for (int w = 0; w < 4; w++) {
            const uint4 bw = __ldg(bp + c * 4 + w);
            const uint32_t b4[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
            for (int k = 0; k < 8; k++) {
              const float bv = bf16_bits_to_float((k & 1) ? (b4[k >> 1] >> 16) : (b4[k >> 1] & 0xFFFFu));
              v[c][8 * w + k] = __float_as_uint(__uint_as_float(v[c][8 * w + k]) + bv);
            }
          }
        }
      }
      const int64_t row0 = T.m0 + 128 * rank + q * 32;
      if (leader || T.upper) {  // an upper half past the expert's segment is not stored
#pragma unroll
        for (int c = 0; c < 4; c++) {
          stage_reuse_wait(lane);
          store_bf16_block(reinterpret_cast<const float*>(v[c]), stg, lane, &tmO, T.n0 + half * 128 + 32 * c, row0);
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores have landed
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_pair_status, DEV_TIMEOUT);
  cluster_sync_all();  // neither CTA frees tensor memory or exits while the other still uses the pair
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" :: "r"(tmem_base) : "memory");
  cluster_sync_all();
}

cudaError_t launch_gemm_pair(const PairParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& to, cudaStream_t s,
                             int num_sms) {
  int64_t pairs = p.num_tiles < num_sms / 2 ? p.num_tiles : num_sms / 2;
  if (pairs < 1) pairs = 1;
  if (p.f4) {
    constexpr int smem = pair::PCfg<true>::SMEM;
    const cudaError_t e = ensure_smem_attr<mx_gemm_pair_kernel<true>>(smem);
    if (e != cudaSuccess) return e;
    mx_gemm_pair_kernel<true><<<(unsigned)(2 * pairs), pair::THREADS, smem, s>>>(ta, tb, tsa, tsb, to, p);
  } else {
    constexpr int smem = pair::PCfg<false>::SMEM;
    const cudaError_t e = ensure_smem_attr<mx_gemm_pair_kernel<false>>(smem);
    if (e != cudaSuccess) return e;
    mx_gemm_pair_kernel<false><<<(unsigned)(2 * pairs), pair::THREADS, smem, s>>>(ta, tb, tsa, tsb, to, p);
  }
  return cudaGetLastError();
}

cudaError_t read_pair_status(unsigned* out) { return cudaMemcpyFromSymbol(out, g_pair_status, sizeof(unsigned)); }
cudaError_t reset_pair_status() {
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_pair_status, &zero, sizeof(unsigned));
}

}  // namespace mx
