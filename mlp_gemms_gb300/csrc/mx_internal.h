// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mx.h"
#include "attr_guard.h"

namespace mx {

inline int64_t round_up_i64(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline size_t scale_bytes(int64_t rows, int64_t scale_cols) {
  return (size_t)(round_up_i64(rows, 128) * round_up_i64(scale_cols, 4));
}
inline int64_t payload_row_bytes(int64_t cols, int fmt) {
  return fmt == 0 ? cols : (fmt == 1 ? cols / 4 * 3 : cols / 2);
}

struct QuantLaunch {
  const void* x;
  int64_t batch, rows, cols, ld;
  int fmt, hadamard;
  uint8_t* row_data;   // null: no rowwise output
  uint8_t* row_scale;
  uint8_t* col_data;   // null: no columnwise output
  uint8_t* col_scale;
  float* colsum_partials;  // null: no column sums
  float* colsum;
  CUtensorMap xmap;        // BF16 [batch*rows, cols], box 64 x 128, 128-byte swizzle
  CUtensorMap rowmap;      // E4M3: row payload [batch*rows, cols] bytes, box 128 x 128, 128-byte swizzle
  CUtensorMap colmap;      // E4M3: col payload [batch*cols, rows] bytes, same boxes
  int num_sms;
  bool stochastic = false; // stochastic rounding of the elements (E2M3, E2M1)
  uint64_t seed = 0;       // its generator key
  // gather (token permute): output row r is x row src[r], zero where
  // src[r] < 0; rows from offsets[G-1] on are not produced
  const int32_t* src = nullptr;
  int64_t src_rows = 0;
  const int32_t* offsets = nullptr;
  int G = 0;
};
cudaError_t launch_quantize(const QuantLaunch& q, cudaStream_t s);
cudaError_t read_quant_status(unsigned* out);
// Capacity (fp32 values) of the fixed column-sum scratch and its address on
// the current device.
constexpr size_t kNoAllocColsumFloats = size_t(1) << 21;
cudaError_t colsum_scratch(float** out, size_t* floats);
cudaError_t reset_quant_status();

enum GemmMode : int { MODE_GROUPED = 0, MODE_WGRAD = 1 };
constexpr int MAX_SPLIT_EXPERTS = 16;  // wgrad K-split: experts split at most (the kernel's MAX_SPLIT)
enum GemmEpi : int { EPI_BF16 = 0, EPI_SWIGLU = 1, EPI_DSWIGLU = 2, EPI_GELU = 3, EPI_DGELU = 4, EPI_F32 = 5 };

// Everything a grouped-GEMM launch needs besides the two tensor maps.
struct GemmParams {
  int mode, epi;
  int G;
  const int32_t* offsets;   // device [G], cumulative segment ends
  int64_t R;                // rows of A (grouped) / reduction extent (wgrad)
  int64_t K;                // reduction length (grouped; multiple of 128)
  int64_t Nb;               // B rows per expert (grouped) / B rows total (wgrad)
  int64_t Mw;               // rows of A (wgrad)
  int64_t F;                // SwiGLU FFN width (FC1 out = 2F)
  int a_type, b_type;       // MMA element types (E4M3 = 0, E2M3 = 3, E2M1 = 5)
  int f4;                   // packed E2M1 operands on .kind::mxf4 (plain epilogues)
  int32_t* dyn_ctr;         // wgrad: tile counter for the dynamic schedule (zeroed by the host), or null
  uint32_t tx_bytes;        // bytes one pipeline stage's copies complete on its barrier
  const uint8_t* sfa;
  const uint8_t* sfb;
  int64_t sfa_kchunks, sfb_kchunks;  // 512-byte chunks per 128-row block
  int m_tiles, n_tiles;
  int64_t num_tiles;
  // epilogue outputs
  uint16_t* out;            // BF16 [rows, out_ld]
  int64_t out_ld;
  uint16_t* z;              // SwiGLU: BF16 pre-activation save [R, 2F]; dSwiGLU: its input
  uint8_t* q_row;           // requantized rowwise payload [R, C]
  uint8_t* q_row_scale;
  uint8_t* q_col;           // requantized columnwise payload [C, R]
  uint8_t* q_col_scale;
  int64_t q_cols;           // C: F (SwiGLU), 2F (dSwiGLU), H (GELU / dGELU)
  int64_t q_row_ld, q_col_ld;  // payload bytes per row of q_row / q_col
  int q_fmt, q_had;         // requant element format and rotation (GELU / dGELU)
  const uint16_t* bias;     // BF16 [N] added to the fp32 accumulator, or null
  int64_t bias_ld;          // grouped: elements between experts' bias rows (0: one row for all)
  float* colsum_partials;   // dGELU: fp32 [ceil(R/128), C] per-tile column sums
  float* tap;               // test instrument: fused epilogues' fp32 pre-quant values [R, C], or null
  float* out_f32;           // EPI_F32: fp32 gradient buffer [rows, out_ld] (wgrad into main_grad)
  int accumulate;           // EPI_F32: 0 stores, 1 adds into what out_f32 holds
  const float* probs;       // SwiGLU / dSwiGLU: routing probability per row [R], or null
  float* dprobs_part;       // dSwiGLU with probs: per-row partial sums [R, dprobs_ld]
  int64_t dprobs_ld;        // 2 per 128-column tile of F
  // wgrad K-split of the largest experts (split_chunks = 0: none; an expert
  // with more than split_min chunks gets parts of at most split_chunks): fp32
  // partial tiles [128][BN] in split_ws (split_slots of them), one arrival
  // counter per split tile in split_cnt (zero before the launch, zero after),
  // at most split_extra extra tiles (the num_tiles headroom)
  int split_chunks;
  int split_min;            // experts with more chunks than this are split
  float* split_ws;
  int32_t* split_cnt;
  int64_t split_slots;
  int64_t split_extra;
};

// ta, tb: operand maps; to: the BF16 output map (32x32 boxes, 64-byte
// swizzle) of the epilogue's BF16 output, or any valid map when it has none.
// Experts the CTA-pair kernels' row-tile table holds (their device constant
// MAX_PAIR_G).
constexpr int MAX_PAIR_G_HOST = 1024;

// The SwiGLU forward / dSwiGLU backward on CTA pairs: tsa / tsb map the
// operands' blocked scales ([row blocks][K chunks][512 B], boxes of one
// chunk of one row block) for the 2-SM scale loads.
cudaError_t launch_gemm_pair_fused(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                                   const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& to,
                                   cudaStream_t s, int num_sms);
cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                        int bn, cudaStream_t s, int num_sms);
cudaError_t launch_gemm_dense(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to, int bn, cudaStream_t s, int num_sms);
cudaError_t launch_colsum_reduce(const float* partials, int64_t tiles, int64_t cols, float* out, cudaStream_t s);
// dprobs[r] = sum over k of part[r, k] in order, for the rows of the segments
// (r < offsets[G-1], or all R rows without offsets); other rows untouched.
cudaError_t launch_dprobs_reduce(const float* part, int64_t R, int64_t ld, const int32_t* offsets, int G,
                                 float* dprobs, cudaStream_t s);
// The CTA-pair grouped GEMM (gemm_pair.cu): 256 x 256 tiles on two SMs,
// BF16 out through a [R, Nb] tensor map; segments multiples of 256 rows.
struct PairParams {
  int G;
  const int32_t* offsets;  // device [G], cumulative segment ends (NULL: one segment of R rows)
  int64_t R, K, Nb;        // A [R, K], B [G * Nb, K]
  int a_type, b_type;      // MMA element types
  int64_t n_tiles, num_tiles;  // 256-column tiles per row block; pair tiles in all
  uint32_t tx_bytes;       // one CTA's bytes per stage (A and B boxes, scale chunks)
  int f4;                  // packed E2M1 operands on .kind::mxf4 (256 K-elements a stage)
  const uint16_t* bias;    // BF16 bias added to the fp32 accumulator before the rounding, or null
  int64_t bias_ld;         // elements between experts' bias rows (0: one row for all)
};
cudaError_t launch_gemm_pair(const PairParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& to, cudaStream_t s,
                             int num_sms);
cudaError_t read_pair_status(unsigned* out);
cudaError_t reset_pair_status();
cudaError_t read_gemm_status(unsigned* out);
cudaError_t reset_gemm_status();
cudaError_t read_dense_status(unsigned* out);
cudaError_t reset_dense_status();
// The BF16 / fp32 epilogues on packed E2M1 operands (.kind::mxf4).
cudaError_t launch_gemm_f4(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                           int bn, cudaStream_t s, int num_sms);
cudaError_t read_f4_status(unsigned* out);
cudaError_t reset_f4_status();
// Token permute support (permute.cu).  counts: the workspace, int32
// [G, ceil(T*k / 1024)] (expert-major).
cudaError_t launch_route_index(const int32_t* topk, int64_t T, int k, int G, int32_t* offsets, int32_t* src,
                               int64_t R_cap, int32_t* row_of, int32_t* counts, int32_t pad, cudaStream_t s);
cudaError_t launch_unpermute(const uint16_t* in, int64_t R, int64_t D, const int32_t* row_of, const float* w,
                             int64_t T, int k, uint16_t* out, int num_sms, cudaStream_t s);
cudaError_t read_perm_status(unsigned* out);
cudaError_t reset_perm_status();
constexpr int kRouteChunk = 1024;
cudaError_t launch_wait_selftest(uint64_t budget_ns, cudaStream_t s);

// The tensors of one MLP step that the host pipeline moves: raw inputs the
// step reads once (X, W1, W2, dY, b1, b2) and outputs it writes (y, dX, dW1,
// dW2, db1, db2).
enum StepTensor { T_X, T_W1, T_W2, T_DY, T_B1, T_B2, T_Y, T_DX, T_DW1, T_DW2, T_DB1, T_DB2, T_COUNT };
inline bool step_tensor_is_input(int t) { return t <= T_B2; }

// Called on the host while a step is being enqueued: before(t) just before
// the launch that reads input t or writes output t, after(t) just after it.
struct StepHooks {
  void (*before)(void* ctx, int t);
  void (*after)(void* ctx, int t);
  void* ctx;
};
mx_status_t mlp_check(const mx_mlp_args_t* a);
// Sets the calling thread's mx_last_error() message; returns st.
mx_status_t set_error(mx_status_t st, const char* msg);
mx_status_t mlp_step(const mx_mlp_args_t* a, mx_stream_t stream, const StepHooks* hooks);

}  // namespace mx
