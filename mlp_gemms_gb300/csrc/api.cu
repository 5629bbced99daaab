// C ABI of the MX training-MLP library: host-side validation, TMA tensor
// maps, launch configuration and the MLP step.  Nothing here allocates
// device memory; every buffer belongs to the caller.
//
// torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
// group gemm": cudnn-fe ops commit (two-tier validation: always-on metadata
// checks plus opt-in value checks of the offsets that need a sync) and the
// hardening commit (int32 element-index guards, 16-byte pointer gate, G == 0
// rejected, R == 0 returns early without a launch).
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/mx.h"
#include "mx_internal.h"

namespace {

thread_local std::string g_last_error;

mx_status_t fail(mx_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mx_status_t fail(mx_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mx_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// The thread's last error message, set from other translation units.
mx_status_t mx::set_error(mx_status_t st, const char* msg) { return fail(st, "%s", msg); }

namespace {

#define MX_CHECK(cond, st, ...) \
  do {                          \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align_up(size_t x) { return (x + 255) / 256 * 256; }

// ---- device properties --------------------------------------------------

struct DevInfo {
  bool known = false;
  int major = 0, minor = 0, sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

mx_status_t device_info(DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MX_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.known) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.known = true;
  }
  *out = d;
  if (d.major != 10 || d.minor != 3)
    return fail(MX_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; this library runs on 10.3 only",
                dev, d.major, d.minor);
  return MX_OK;
}

// ---- TMA tensor maps ----------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

mx_status_t get_encoder() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  return MX_OK;
}

// 2-D MX payload [rows, K elements] as a TMA tensor, box 128 elements x 128
// rows with the 128-byte swizzle.  E4M3 is plain bytes; E2M3 and E2M1 use
// the packed sub-byte types, which expand each 16-element group into a
// 16-byte shared-memory slot -- the operand form the block-scaled MMA reads.
mx_status_t make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int fmt) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  CUtensorMapDataType dt = fmt == MX_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : (fmt == MX_E2M3 ? CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B
                                             : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B);
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)mx::payload_row_bytes(k, fmt)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MX_OK;
}

// Packed E2M1 payload [rows, K elements] as bytes (two elements each) for
// .kind::mxf4: box 128 bytes (256 elements) x 128 rows, 128-byte swizzle.
mx_status_t make_tmap_packed(CUtensorMap* m, const void* base, int64_t rows, int64_t k) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (packed E2M1) failed (%d)", (int)r);
  return MX_OK;
}

// BF16 input [rows, cols] with row stride ld elements: boxes of 64 columns
// x 128 rows with the 128-byte swizzle (two per 128x128 quantizer tile, or
// the z slots of the 128-column dSwiGLU tiles), or of 32 columns with the
// 64-byte swizzle and 64-byte L2 fetches (the 256-column dSwiGLU tiles' z
// slots).
mx_status_t make_tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
                           int box_cols = 64) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        box_cols == 32 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (input) failed (%d)", (int)r);
  return MX_OK;
}

// BF16 output [rows, cols] with row stride ld elements as TMA store
// target: 32x32 boxes, 64-byte swizzle (matching the epilogue's staging).
mx_status_t make_tmap_out(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
  return MX_OK;
}

// fp32 output [rows, cols] with row stride ld elements as TMA store or
// reduce-add target: 16x32 boxes (64-byte rows), 64-byte swizzle.
mx_status_t make_tmap_out_f32(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (fp32 output) failed (%d)", (int)r);
  return MX_OK;
}

// Blocked scales of a [rows, K] MX tensor as [row blocks][K chunks][512
// bytes] (64 x 8-byte elements per chunk), boxes of `chunks` consecutive
// chunks x `blocks` consecutive row blocks: the CTA-pair GEMM loads a
// stage's scale chunks with the 2-SM TMA form.
mx_status_t make_tmap_scales(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int blocks, int chunks) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  const int64_t kchunks = (k / 32 + 3) / 4, rblocks = (rows + 127) / 128;
  cuuint64_t dims[3] = {64, (cuuint64_t)kchunks, (cuuint64_t)rblocks};
  cuuint64_t strides[2] = {512, (cuuint64_t)(kchunks * 512)};
  cuuint32_t box[3] = {64, (cuuint32_t)chunks, (cuuint32_t)blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", (int)r);
  return MX_OK;
}

// Byte tensor [rows, row_bytes] as a TMA store target: box 128 bytes x 128
// rows, 128-byte swizzle (the quantizer's staging layout).
mx_status_t make_tmap_bytes(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_bytes) {
  mx_status_t st = get_encoder();
  if (st != MX_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_bytes, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled (payload) failed (%d)", (int)r);
  return MX_OK;
}

// The quantizer stages E4M3 and E2M1 tiles in shared memory and stores
// them with TMA: box 128 bytes (E4M3, 128 elements) or 64 bytes (E2M1).
bool staged(int fmt) { return fmt == MX_E4M3 || fmt == MX_E2M1; }
int staged_box(int fmt) { return fmt == MX_E4M3 ? 128 : 64; }

// tcgen05 .kind::mxf8f6f4 element type code of an MX format.
int mma_type(int fmt) { return fmt == MX_E4M3 ? 0 : (fmt == MX_E2M3 ? 3 : 5); }

// ---- argument checks ----------------------------------------------------

mx_status_t check_tensor(const mx_tensor_t* t, const char* name, int64_t rows, int64_t cols, int fmt, int had) {
  MX_CHECK(t != nullptr, MX_ERR_INVALID_ARG, "%s is NULL", name);
  MX_CHECK(t->rows == rows && t->cols == cols, MX_ERR_SHAPE, "%s is [%lld, %lld], expected [%lld, %lld]", name,
           (long long)t->rows, (long long)t->cols, (long long)rows, (long long)cols);
  if (rows == 0 || cols == 0) return MX_OK;  // empty: no storage to check
  MX_CHECK(t->data != nullptr && t->scale != nullptr, MX_ERR_INVALID_ARG, "%s has a NULL data or scale pointer", name);
  MX_CHECK(t->fmt == fmt, MX_ERR_INVALID_ARG, "%s has format %d, expected %d", name, t->fmt, fmt);
  MX_CHECK((t->hadamard != 0) == (had != 0), MX_ERR_INVALID_ARG, "%s rotation flag %d, expected %d", name,
           t->hadamard, had);
  MX_CHECK(aligned16(t->data) && aligned16(t->scale), MX_ERR_ALIGNMENT, "%s pointers must be 16-byte aligned", name);
  return MX_OK;
}

mx_status_t check_gemm_operand(const mx_tensor_t* t, const char* name) {
  MX_CHECK(t != nullptr, MX_ERR_INVALID_ARG, "%s is NULL", name);
  MX_CHECK(t->rows >= 0 && t->cols > 0, MX_ERR_SHAPE, "%s has shape [%lld, %lld]", name, (long long)t->rows,
           (long long)t->cols);
  if (t->rows > 0) {
    MX_CHECK(t->data != nullptr && t->scale != nullptr, MX_ERR_INVALID_ARG, "%s has a NULL data or scale pointer",
             name);
    MX_CHECK(aligned16(t->data) && aligned16(t->scale), MX_ERR_ALIGNMENT, "%s pointers must be 16-byte aligned",
             name);
  }
  MX_CHECK(t->fmt >= MX_E4M3 && t->fmt <= MX_E2M1, MX_ERR_INVALID_ARG, "%s has format %d", name, t->fmt);
  // the packed sub-byte tensor-map types need 32-byte aligned rows
  MX_CHECK(t->fmt == MX_E4M3 || (reinterpret_cast<uintptr_t>(t->data) & 31u) == 0, MX_ERR_ALIGNMENT,
           "%s: E2M3/E2M1 payload must be 32-byte aligned", name);
  MX_CHECK(t->rows < (1ll << 31) && t->cols < (1ll << 31), MX_ERR_SHAPE, "%s exceeds the int32 coordinate range", name);
  return MX_OK;
}

mx_status_t check_pair(const mx_tensor_t* a, const mx_tensor_t* b, const char* an, const char* bn) {
  MX_CHECK(a->fmt == b->fmt, MX_ERR_INVALID_ARG, "%s and %s have different formats (%d, %d)", an, bn, a->fmt, b->fmt);
  MX_CHECK((a->hadamard != 0) == (b->hadamard != 0), MX_ERR_INVALID_ARG,
           "%s and %s must both carry the rotation or neither", an, bn);
  MX_CHECK(a->fmt == MX_E4M3 || a->cols % 128 == 0, MX_ERR_SHAPE, "packed operands need K %% 128 == 0");
  return MX_OK;
}

bool env_validate_offsets() {
  const char* v = getenv("MX_VALIDATE_OFFSETS");
  return v && v[0] == '1';
}

// MX_LOG=1: one line on stderr for each launch configuration the process
// has not launched before (kernel, epilogue, tile width, shapes, grid), read
// from the environment once.  The configurations seen are kept in a set of
// at most 4096 entries (past that, nothing more is printed).
bool env_log() {
  static const bool on = [] {
    const char* v = getenv("MX_LOG");
    return v && v[0] == '1';
  }();
  return on;
}

void log_config(const char* fmt, ...) {
  if (!env_log()) return;
  char line[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(line, sizeof(line), fmt, ap);
  va_end(ap);
  static std::mutex mu;
  static std::unordered_set<std::string> seen;
  std::lock_guard<std::mutex> lk(mu);
  if (seen.size() >= 4096 || !seen.insert(line).second) return;
  fprintf(stderr, "mx: %s\n", line);
}

const char* epi_name(int epi) {
  static const char* names[] = {"bf16", "swiglu", "dswiglu", "gelu", "dgelu", "f32"};
  return (epi >= 0 && epi <= 5) ? names[epi] : "?";
}

// Opt-in value check of the offsets (synchronises the stream).
mx_status_t validate_offsets_values(const int32_t* offsets_dev, int G, int64_t R, cudaStream_t s) {
  std::vector<int32_t> h((size_t)G);
  cudaError_t e = cudaMemcpyAsync(h.data(), offsets_dev, sizeof(int32_t) * (size_t)G, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading offsets");
  int64_t prev = 0;
  for (int g = 0; g < G; g++) {
    MX_CHECK(h[g] % 128 == 0, MX_ERR_OFFSETS, "offsets[%d] = %d is not a multiple of 128", g, h[g]);
    MX_CHECK(h[g] >= prev, MX_ERR_OFFSETS, "offsets[%d] = %d decreases (previous %lld)", g, h[g], (long long)prev);
    prev = h[g];
  }
  MX_CHECK(prev <= R, MX_ERR_OFFSETS, "offsets[G-1] = %lld exceeds R = %lld", (long long)prev, (long long)R);
  return MX_OK;
}

mx_status_t check_offsets(const int32_t* offsets, int32_t G, int64_t R, cudaStream_t s) {
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  if (offsets == nullptr && G == 1) return MX_OK;  // one segment of all rows
  MX_CHECK(offsets != nullptr, MX_ERR_INVALID_ARG, "offsets is NULL");
  MX_CHECK((reinterpret_cast<uintptr_t>(offsets) & 3u) == 0, MX_ERR_ALIGNMENT, "offsets must be 4-byte aligned");
  if (env_validate_offsets()) return validate_offsets_values(offsets, G, R, s);
  return MX_OK;
}

// Bytes one pipeline stage completes on its barrier: the A box (128 rows),
// the B boxes (bn rows) and the scale chunks.  For the packed sub-byte types
// the tensor copy counts the packed data, 128 elements a row.
uint32_t stage_tx_bytes(int fmt, int bn) {
  const uint32_t row = (uint32_t)mx::payload_row_bytes(128, fmt);
  return (128u + (uint32_t)bn) * row + 512u + (uint32_t)(bn / 128) * 512u;
}

// Test instrument (mx_debug_tap): where the fused epilogues also write
// their fp32 pre-quantization values, per calling thread.
thread_local float* g_tap = nullptr;
thread_local int64_t g_tap_elems = 0;

mx_status_t attach_tap(mx::GemmParams* p, int64_t rows, int64_t cols) {
  if (g_tap == nullptr) return MX_OK;
  MX_CHECK(g_tap_elems >= rows * cols, MX_ERR_SHAPE, "debug tap holds %lld floats, the epilogue writes %lld",
           (long long)g_tap_elems, (long long)(rows * cols));
  p->tap = g_tap;
  return MX_OK;
}

// A BF16 output the epilogue writes with TMA stores (base NULL: none).
struct OutView {
  const void* base;
  int64_t rows, cols, ld;
  bool f32 = false;  // fp32 elements (EPI_F32) instead of BF16
};

// Which fused-epilogue and weight-gradient launches run on CTA pairs (the
// outputs are the same bit for bit either way).  By default only the SwiGLU
// forward (0.73 -> 0.69-0.70 ms: its mainloop is the limit); the dSwiGLU
// backward is bound by its epilogue (0.63 on one SM per tile, 0.66 on
// pairs) and the weight gradients lose on pairs (dW1 0.70 -> 0.75 ms: half
// as many units of twice the work for the claimed-tile balance under the
// skewed routing).  MX_FUSED_PAIRS=0 keeps all on one SM per tile,
// MX_FUSED_PAIRS=1 puts all on pairs.  Read at every call.
bool fused_pairs_enabled(bool by_default) {
  const char* v = getenv("MX_FUSED_PAIRS");
  if (v && v[0] == '0') return false;
  if (v && v[0] == '1') return true;
  return by_default;
}

mx_status_t run_gemm(mx::GemmParams p, const mx_tensor_t* a, const mx_tensor_t* b, int bn, cudaStream_t s,
                     const DevInfo& dev, OutView out, bool pair = false) {
  // E2M1 operands with a plain epilogue run on .kind::mxf4 from the packed
  // payload; the fused epilogues keep .kind::mxf8f6f4.
  p.f4 = (a->fmt == MX_E2M1 && (p.epi == mx::EPI_BF16 || p.epi == mx::EPI_F32)) ? 1 : 0;
  p.tx_bytes = stage_tx_bytes(a->fmt, bn);
  CUtensorMap ta, tb, to;
  mx_status_t st = p.f4 ? make_tmap_packed(&ta, a->data, a->rows, a->cols)
                        : make_tmap(&ta, a->data, a->rows, a->cols, a->fmt);
  if (st != MX_OK) return st;
  if ((st = p.f4 ? make_tmap_packed(&tb, b->data, b->rows, b->cols)
                 : make_tmap(&tb, b->data, b->rows, b->cols, b->fmt)) != MX_OK)
    return st;
  if (out.base) {
    st = out.f32 ? make_tmap_out_f32(&to, out.base, out.rows, out.cols, out.ld)
                 : make_tmap_out(&to, out.base, out.rows, out.cols, out.ld);
    if (st != MX_OK) return st;
  } else if (p.epi == mx::EPI_DSWIGLU) {  // the saved z [R, 2F], streamed by the epilogue (64 / 32 columns a box)
    if ((st = make_tmap_bf16(&to, p.z, p.R, 2 * p.F, 2 * p.F, bn == 256 ? 32 : 64)) != MX_OK) return st;
  } else {
    to = ta;
  }
  if (pair) {
    // CTA pairs: 256-row tiles per expert segment (the last one of an odd
    // 128-row block count half computed past the segment), each CTA staging
    // its 128 A rows, one 128-row block of B and the scale chunks of its A
    // rows and of both B blocks
    p.tx_bytes = stage_tx_bytes(a->fmt, 128) + 512u;
    if (p.mode == mx::MODE_GROUPED) p.num_tiles = ((p.R + 255) / 256 + (p.offsets ? (p.G + 1) / 2 : 0)) * p.n_tiles;
    CUtensorMap tsa, tsb;
    if ((st = make_tmap_scales(&tsa, a->scale, a->rows, a->cols, 1, 1)) != MX_OK) return st;
    if ((st = make_tmap_scales(&tsb, b->scale, b->rows, b->cols, 1, 1)) != MX_OK) return st;
    log_config("gemm pair %s BN=256 a=%d b=%d R=%lld K=%lld N=%lld G=%d tiles=%lld", epi_name(p.epi), p.a_type,
               p.b_type, (long long)p.R, (long long)p.K, (long long)p.Nb, p.G, (long long)p.num_tiles);
    cudaError_t e = mx::launch_gemm_pair_fused(p, ta, tb, tsa, tsb, to, s, dev.sms);
    if (e != cudaSuccess) return cuda_fail(e, "CTA-pair fused GEMM launch");
    return MX_OK;
  }
  log_config("gemm %s %s%s BN=%d a=%d b=%d R=%lld K=%lld N=%lld G=%d tiles=%lld grid=%lld split=%d",
             p.mode == mx::MODE_WGRAD ? "wgrad" : "grouped", epi_name(p.epi), p.f4 ? " mxf4" : "", bn, p.a_type,
             p.b_type, (long long)p.R, (long long)p.K, (long long)p.Nb, p.G, (long long)p.num_tiles,
             (long long)(p.num_tiles < dev.sms ? p.num_tiles : dev.sms), p.split_chunks > 0 ? 1 : 0);
  cudaError_t e = mx::launch_gemm(p, ta, tb, to, bn, s, dev.sms);
  if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM launch");
  return MX_OK;
}

mx::GemmParams base_params() {
  mx::GemmParams p;
  memset(&p, 0, sizeof(p));
  return p;
}

}  // namespace

extern "C" {

int mx_abi_version(void) { return MX_ABI_VERSION; }

const char* mx_last_error(void) { return g_last_error.c_str(); }

const char* mx_status_string(mx_status_t st) {
  switch (st) {
    case MX_OK: return "ok";
    case MX_ERR_INVALID_ARG: return "invalid argument";
    case MX_ERR_SHAPE: return "bad shape";
    case MX_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case MX_ERR_OFFSETS: return "malformed offsets";
    case MX_ERR_UNSUPPORTED_DEVICE: return "unsupported device";
    case MX_ERR_CUDA: return "CUDA error";
    case MX_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MX_ERR_WORKSPACE: return "workspace too small";
    case MX_ERR_NOT_SUPPORTED: return "not supported";
  }
  return "unknown status";
}

size_t mx_payload_bytes(int64_t rows, int64_t cols, int32_t fmt) {
  if (rows < 0 || cols < 0 || fmt < 0 || fmt > 2) return 0;
  return (size_t)(rows * mx::payload_row_bytes(cols, fmt));
}

size_t mx_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return mx::scale_bytes(rows, cols / 32);
}

size_t mx_quantize_workspace_bytes(int64_t rows, int64_t cols, uint32_t flags) {
  if (!(flags & MX_COLSUM) || rows <= 0 || cols <= 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)cols * sizeof(float);
}

}  // extern "C"

namespace {

mx_status_t quantize_impl(const void* x_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t ld, int32_t fmt,
                          uint32_t flags, const mx_tensor_t* out_row, const mx_tensor_t* out_col, float* colsum,
                          void* workspace, size_t workspace_bytes, bool stochastic, uint64_t seed,
                          mx_stream_t stream) {
  MX_CHECK(fmt >= MX_E4M3 && fmt <= MX_E2M1, MX_ERR_INVALID_ARG, "fmt = %d is not an MX element format", fmt);
  MX_CHECK((flags & ~0xFu) == 0, MX_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  MX_CHECK(flags & (MX_ROWWISE | MX_COLWISE), MX_ERR_INVALID_ARG, "neither MX_ROWWISE nor MX_COLWISE requested");
  MX_CHECK(batch >= 1, MX_ERR_SHAPE, "batch = %lld", (long long)batch);
  MX_CHECK(rows >= 0 && cols > 0, MX_ERR_SHAPE, "shape [%lld, %lld]", (long long)rows, (long long)cols);
  MX_CHECK(cols % 32 == 0, MX_ERR_SHAPE, "cols = %lld is not a multiple of 32", (long long)cols);
  MX_CHECK(!(flags & MX_COLWISE) || rows % 32 == 0, MX_ERR_SHAPE, "columnwise needs rows %% 32 == 0 (rows = %lld)",
           (long long)rows);
  MX_CHECK(batch == 1 || (rows % 128 == 0 && cols % 128 == 0), MX_ERR_SHAPE,
           "batched quantization needs rows and cols multiples of 128");
  MX_CHECK(ld >= cols && ld % 8 == 0, MX_ERR_ALIGNMENT, "ld = %lld must be >= cols and a multiple of 8",
           (long long)ld);
  MX_CHECK(rows == 0 || x_bf16 != nullptr, MX_ERR_INVALID_ARG, "x is NULL");
  MX_CHECK(aligned16(x_bf16), MX_ERR_ALIGNMENT, "x must be 16-byte aligned");
  // bound each factor before multiplying, so no product below can overflow
  MX_CHECK(rows < (1ll << 31) && batch < (1ll << 31) && ld < (1ll << 40), MX_ERR_SHAPE, "input too large");
  MX_CHECK(rows * batch < (1ll << 31) && (rows == 0 || ld <= ((1ll << 40) - 1) / (rows * batch)), MX_ERR_SHAPE,
           "input too large");
  const int had = (flags & MX_HADAMARD) ? 1 : 0;
  mx_status_t st;
  if (flags & MX_ROWWISE) {
    if ((st = check_tensor(out_row, "out_row", batch * rows, cols, fmt, had)) != MX_OK) return st;
  }
  if (flags & MX_COLWISE) {
    if ((st = check_tensor(out_col, "out_col", batch * cols, rows, fmt, had)) != MX_OK) return st;
  }
  if (flags & MX_COLSUM) {
    MX_CHECK(flags & MX_COLWISE, MX_ERR_INVALID_ARG, "MX_COLSUM needs MX_COLWISE");
    MX_CHECK(batch == 1, MX_ERR_INVALID_ARG, "MX_COLSUM needs batch == 1");
    MX_CHECK(colsum != nullptr && aligned16(colsum), MX_ERR_INVALID_ARG, "colsum must be a 16-byte aligned pointer");
    const size_t need = mx_quantize_workspace_bytes(rows, cols, flags);
    MX_CHECK(need == 0 || (workspace != nullptr && aligned16(workspace) && workspace_bytes >= need),
             MX_ERR_WORKSPACE, "MX_COLSUM needs %zu bytes of 16-byte aligned workspace", need);
  }
  if (rows == 0) {
    // no rows: nothing to quantize; each column's sum over zero rows is 0
    if (flags & MX_COLSUM) {
      cudaError_t e = cudaMemsetAsync(colsum, 0, (size_t)cols * sizeof(float), reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "clearing colsum");
    }
    return MX_OK;
  }
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::QuantLaunch q;
  q.x = x_bf16;
  q.batch = batch; q.rows = rows; q.cols = cols; q.ld = ld;
  q.fmt = fmt; q.hadamard = had;
  q.row_data = (flags & MX_ROWWISE) ? static_cast<uint8_t*>(out_row->data) : nullptr;
  q.row_scale = (flags & MX_ROWWISE) ? out_row->scale : nullptr;
  q.col_data = (flags & MX_COLWISE) ? static_cast<uint8_t*>(out_col->data) : nullptr;
  q.col_scale = (flags & MX_COLWISE) ? out_col->scale : nullptr;
  q.colsum_partials = (flags & MX_COLSUM) ? static_cast<float*>(workspace) : nullptr;
  q.colsum = colsum;
  q.num_sms = dev.sms;
  q.stochastic = stochastic;
  q.seed = seed;
  if ((st = make_tmap_bf16(&q.xmap, x_bf16, batch * rows, cols, ld)) != MX_OK) return st;
  q.rowmap = q.colmap = q.xmap;  // placeholders where no staged store is made
  if (staged(fmt) && (flags & MX_ROWWISE)) {
    if ((st = make_tmap_bytes(&q.rowmap, out_row->data, batch * rows, mx::payload_row_bytes(cols, fmt),
                              staged_box(fmt))) != MX_OK)
      return st;
  }
  if (staged(fmt) && (flags & MX_COLWISE)) {
    if ((st = make_tmap_bytes(&q.colmap, out_col->data, batch * cols, mx::payload_row_bytes(rows, fmt),
                              staged_box(fmt))) != MX_OK)
      return st;
  }
  log_config("quantize fmt=%d flags=0x%x%s batch=%lld rows=%lld cols=%lld", fmt, flags, stochastic ? " sr" : "",
             (long long)batch, (long long)rows, (long long)cols);
  cudaError_t e = mx::launch_quantize(q, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return MX_OK;
}

}  // namespace

extern "C" {

mx_status_t mx_quantize(const void* x_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t ld, int32_t fmt,
                        uint32_t flags, const mx_tensor_t* out_row, const mx_tensor_t* out_col, float* colsum,
                        void* workspace, size_t workspace_bytes, mx_stream_t stream) {
  return quantize_impl(x_bf16, batch, rows, cols, ld, fmt, flags, out_row, out_col, colsum, workspace,
                       workspace_bytes, false, 0, stream);
}

mx_status_t mx_quantize_sr(const void* x_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t ld, int32_t fmt,
                           uint32_t flags, uint64_t seed, const mx_tensor_t* out_row, const mx_tensor_t* out_col,
                           mx_stream_t stream) {
  MX_CHECK(fmt == MX_E2M3 || fmt == MX_E2M1, MX_ERR_NOT_SUPPORTED,
           "stochastic rounding is built for the E2M3 and E2M1 element formats (fmt = %d)", fmt);
  MX_CHECK((flags & MX_COLSUM) == 0, MX_ERR_NOT_SUPPORTED, "MX_COLSUM is not combined with stochastic rounding");
  return quantize_impl(x_bf16, batch, rows, cols, ld, fmt, flags, out_row, out_col, nullptr, nullptr, 0, true, seed,
                       stream);
}

int64_t mx_moe_route_rows_pad(int64_t T, int32_t k, int32_t G, int32_t pad) {
  if (T < 0 || k < 0 || G < 0 || (pad != 128 && pad != 256)) return 0;
  return (T * k + (int64_t)(pad - 1) * G + pad - 1) / pad * pad;
}

int64_t mx_moe_route_rows(int64_t T, int32_t k, int32_t G) { return mx_moe_route_rows_pad(T, k, G, 128); }

size_t mx_moe_route_workspace_bytes(int64_t T, int32_t k, int32_t G) {
  if (T < 0 || k < 0 || G < 0) return 0;
  const int64_t chunks = (T * k + mx::kRouteChunk - 1) / mx::kRouteChunk;
  return (size_t)(chunks > 0 ? chunks : 1) * (size_t)G * sizeof(int32_t);
}

mx_status_t mx_moe_route_index(const int32_t* topk_dev, int64_t T, int32_t k, int32_t G, int32_t* offsets_dev,
                               int32_t* src_dev, int64_t R_cap, int32_t* row_of_dev, void* workspace,
                               size_t workspace_bytes, mx_stream_t stream) {
  return mx_moe_route_index_pad(topk_dev, T, k, G, 128, offsets_dev, src_dev, R_cap, row_of_dev, workspace,
                                workspace_bytes, stream);
}

mx_status_t mx_moe_route_index_pad(const int32_t* topk_dev, int64_t T, int32_t k, int32_t G, int32_t pad,
                                   int32_t* offsets_dev, int32_t* src_dev, int64_t R_cap, int32_t* row_of_dev,
                                   void* workspace, size_t workspace_bytes, mx_stream_t stream) {
  MX_CHECK(pad == 128 || pad == 256, MX_ERR_INVALID_ARG, "pad = %d; segments are padded to 128 or 256 rows", pad);
  MX_CHECK(T >= 0 && k >= 1, MX_ERR_INVALID_ARG, "T = %lld, k = %d", (long long)T, k);
  MX_CHECK(G >= 1 && G <= 1024, MX_ERR_INVALID_ARG, "G = %d is outside [1, 1024]", G);
  MX_CHECK(T * k < (1ll << 31), MX_ERR_SHAPE, "T * k = %lld exceeds the int32 row range", (long long)(T * k));
  MX_CHECK(R_cap >= mx_moe_route_rows_pad(T, k, G, pad) && R_cap < (1ll << 31), MX_ERR_SHAPE,
           "R_cap = %lld; mx_moe_route_rows_pad gives %lld", (long long)R_cap,
           (long long)mx_moe_route_rows_pad(T, k, G, pad));
  MX_CHECK(offsets_dev != nullptr && src_dev != nullptr, MX_ERR_INVALID_ARG, "offsets or src is NULL");
  MX_CHECK(T == 0 || (topk_dev != nullptr && row_of_dev != nullptr), MX_ERR_INVALID_ARG, "topk or row_of is NULL");
  MX_CHECK(aligned16(topk_dev) && aligned16(offsets_dev) && aligned16(src_dev) && aligned16(row_of_dev),
           MX_ERR_ALIGNMENT, "pointers must be 16-byte aligned");
  MX_CHECK(workspace != nullptr && aligned16(workspace) && workspace_bytes >= mx_moe_route_workspace_bytes(T, k, G),
           MX_ERR_WORKSPACE, "mx_moe_route_index needs %zu bytes of 16-byte aligned workspace",
           mx_moe_route_workspace_bytes(T, k, G));
  DevInfo dev;
  mx_status_t st;
  if ((st = device_info(&dev)) != MX_OK) return st;
  cudaError_t e = mx::launch_route_index(topk_dev, T, k, G, offsets_dev, src_dev, R_cap, row_of_dev,
                                         static_cast<int32_t*>(workspace), pad, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "routing index launch");
  return MX_OK;
}

mx_status_t mx_permute_quantize(const void* x_bf16, int64_t T, int64_t D, int64_t ld, const int32_t* src_dev,
                                int64_t R_cap, const int32_t* offsets_dev, int32_t G, int32_t fmt, uint32_t flags,
                                const mx_tensor_t* out_row, const mx_tensor_t* out_col, mx_stream_t stream) {
  MX_CHECK(fmt >= MX_E4M3 && fmt <= MX_E2M1, MX_ERR_INVALID_ARG, "fmt = %d is not an MX element format", fmt);
  MX_CHECK((flags & ~(uint32_t)(MX_ROWWISE | MX_COLWISE)) == 0, MX_ERR_NOT_SUPPORTED,
           "the quantizing permute takes MX_ROWWISE / MX_COLWISE only (flags 0x%x)", flags);
  MX_CHECK(flags & (MX_ROWWISE | MX_COLWISE), MX_ERR_INVALID_ARG, "neither MX_ROWWISE nor MX_COLWISE requested");
  MX_CHECK(T >= 0 && D > 0 && D % 32 == 0, MX_ERR_SHAPE, "T = %lld, D = %lld (D %% 32 == 0)", (long long)T,
           (long long)D);
  MX_CHECK(R_cap >= 0 && R_cap % 128 == 0 && R_cap < (1ll << 31), MX_ERR_SHAPE,
           "R_cap = %lld is not a multiple of 128", (long long)R_cap);
  MX_CHECK(ld >= D && ld % 8 == 0, MX_ERR_ALIGNMENT, "ld = %lld must be >= D and a multiple of 8", (long long)ld);
  MX_CHECK(T == 0 || x_bf16 != nullptr, MX_ERR_INVALID_ARG, "x is NULL");
  MX_CHECK(src_dev != nullptr || R_cap == 0, MX_ERR_INVALID_ARG, "src is NULL");
  MX_CHECK(aligned16(x_bf16) && aligned16(src_dev) && aligned16(offsets_dev), MX_ERR_ALIGNMENT,
           "pointers must be 16-byte aligned");
  MX_CHECK(offsets_dev == nullptr || G >= 1, MX_ERR_INVALID_ARG, "G = %d with offsets", G);
  MX_CHECK(T * ld < (1ll << 40), MX_ERR_SHAPE, "input too large");
  mx_status_t st;
  if (flags & MX_ROWWISE) {
    if ((st = check_tensor(out_row, "out_row", R_cap, D, fmt, 0)) != MX_OK) return st;
  }
  if (flags & MX_COLWISE) {
    if ((st = check_tensor(out_col, "out_col", D, R_cap, fmt, 0)) != MX_OK) return st;
  }
  if (R_cap == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::QuantLaunch q;
  q.x = T > 0 ? x_bf16 : (flags & MX_ROWWISE ? out_row->data : out_col->data);  // never read when T == 0
  q.batch = 1; q.rows = R_cap; q.cols = D; q.ld = ld;
  q.fmt = fmt; q.hadamard = 0;
  q.row_data = (flags & MX_ROWWISE) ? static_cast<uint8_t*>(out_row->data) : nullptr;
  q.row_scale = (flags & MX_ROWWISE) ? out_row->scale : nullptr;
  q.col_data = (flags & MX_COLWISE) ? static_cast<uint8_t*>(out_col->data) : nullptr;
  q.col_scale = (flags & MX_COLWISE) ? out_col->scale : nullptr;
  q.colsum_partials = nullptr;
  q.colsum = nullptr;
  q.num_sms = dev.sms;
  q.src = src_dev; q.src_rows = T; q.offsets = offsets_dev; q.G = G;
  // the gather form reads x with plain copies; the map is an unused kernel argument
  if (T > 0) {
    if ((st = make_tmap_bf16(&q.xmap, x_bf16, T, D, ld)) != MX_OK) return st;
  } else if ((st = make_tmap_bytes(&q.xmap, q.row_data ? q.row_data : q.col_data, 128, 128, 128)) != MX_OK) {
    return st;
  }
  q.rowmap = q.colmap = q.xmap;
  if (staged(fmt) && (flags & MX_ROWWISE)) {
    if ((st = make_tmap_bytes(&q.rowmap, out_row->data, R_cap, mx::payload_row_bytes(D, fmt), staged_box(fmt))) !=
        MX_OK)
      return st;
  }
  if (staged(fmt) && (flags & MX_COLWISE)) {
    if ((st = make_tmap_bytes(&q.colmap, out_col->data, D, mx::payload_row_bytes(R_cap, fmt), staged_box(fmt))) !=
        MX_OK)
      return st;
  }
  cudaError_t e = mx::launch_quantize(q, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantizing permute launch");
  return MX_OK;
}

mx_status_t mx_moe_unpermute(const void* in_bf16, int64_t R, int64_t D, const int32_t* row_of_dev,
                             const float* weights_dev, int64_t T, int32_t k, void* out_bf16, mx_stream_t stream) {
  MX_CHECK(R >= 0 && T >= 0 && k >= 1, MX_ERR_INVALID_ARG, "R = %lld, T = %lld, k = %d", (long long)R, (long long)T, k);
  MX_CHECK(D > 0 && D % 8 == 0, MX_ERR_SHAPE, "D = %lld is not a positive multiple of 8", (long long)D);
  MX_CHECK(T == 0 || (in_bf16 != nullptr || R == 0) && row_of_dev != nullptr && out_bf16 != nullptr,
           MX_ERR_INVALID_ARG, "in, row_of or out is NULL");
  MX_CHECK(aligned16(in_bf16) && aligned16(row_of_dev) && aligned16(weights_dev) && aligned16(out_bf16),
           MX_ERR_ALIGNMENT, "pointers must be 16-byte aligned");
  MX_CHECK(R * D < (1ll << 40) && T * D < (1ll << 40) && T * k < (1ll << 31), MX_ERR_SHAPE, "input too large");
  if (T == 0) return MX_OK;
  DevInfo dev;
  mx_status_t st;
  if ((st = device_info(&dev)) != MX_OK) return st;
  cudaError_t e = mx::launch_unpermute(static_cast<const uint16_t*>(in_bf16), R, D, row_of_dev, weights_dev, T, k,
                                       static_cast<uint16_t*>(out_bf16), dev.sms,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "un-permute launch");
  return MX_OK;
}

mx_status_t mx_quantize_colsum_noalloc(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, int32_t fmt,
                                       uint32_t flags, const mx_tensor_t* out_row, const mx_tensor_t* out_col,
                                       float* colsum, mx_stream_t stream) {
  MX_CHECK((flags & MX_COLSUM) && (flags & MX_COLWISE), MX_ERR_INVALID_ARG,
           "mx_quantize_colsum_noalloc computes column sums: flags need MX_COLSUM and MX_COLWISE");
  MX_CHECK(rows >= 0 && cols > 0, MX_ERR_SHAPE, "shape [%lld, %lld]", (long long)rows, (long long)cols);
  // rows and cols bounded first, so the product cannot wrap past the limit
  const bool fits = rows <= 128 * (int64_t)mx::kNoAllocColsumFloats && cols <= (int64_t)mx::kNoAllocColsumFloats &&
                    (size_t)((rows + 127) / 128) * (size_t)cols <= mx::kNoAllocColsumFloats;
  MX_CHECK(fits, MX_ERR_WORKSPACE,
           "ceil(rows/128) * cols for [%lld, %lld] exceeds the fixed column-sum scratch of %zu values; "
           "use mx_quantize with a workspace", (long long)rows, (long long)cols, mx::kNoAllocColsumFloats);
  float* scratch = nullptr;
  size_t cap = 0;
  cudaError_t e = mx::colsum_scratch(&scratch, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "looking up the column-sum scratch");
  return mx_quantize(x_bf16, 1, rows, cols, ld, fmt, flags, out_row, out_col, colsum, scratch, cap * sizeof(float),
                     stream);
}

}  // extern "C"

namespace {

// The BF16-out grouped GEMM, optionally with expert g's bias row
// bias[g * N .. + N) added to the fp32 accumulator.
mx_status_t grouped_gemm_impl(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                              const void* bias_bf16, void* out_bf16, int64_t ld_out, mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(a, "a")) != MX_OK) return st;
  if ((st = check_gemm_operand(b, "b")) != MX_OK) return st;
  if ((st = check_pair(a, b, "a", "b")) != MX_OK) return st;
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  MX_CHECK(a->cols == b->cols, MX_ERR_SHAPE, "a has K = %lld, b has K = %lld", (long long)a->cols, (long long)b->cols);
  const int64_t K = a->cols, R = a->rows;
  MX_CHECK(K % 128 == 0, MX_ERR_SHAPE, "K = %lld is not a multiple of 128", (long long)K);
  MX_CHECK(b->rows % G == 0, MX_ERR_SHAPE, "b has %lld rows, not a multiple of G = %d", (long long)b->rows, G);
  const int64_t N = b->rows / G;
  MX_CHECK(N > 0 && N % 128 == 0, MX_ERR_SHAPE, "N = %lld per expert is not a positive multiple of 128", (long long)N);
  MX_CHECK(R == 0 || (out_bf16 != nullptr && aligned16(out_bf16)), MX_ERR_ALIGNMENT,
           "out must be a 16-byte aligned pointer");
  MX_CHECK(ld_out >= N && ld_out % 8 == 0, MX_ERR_ALIGNMENT, "ld_out = %lld must be >= N and a multiple of 8",
           (long long)ld_out);
  MX_CHECK(R * ld_out < (1ll << 40), MX_ERR_SHAPE, "output too large");
  if ((st = check_offsets(offsets_dev, G, R, s)) != MX_OK) return st;
  if (R == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  const int bn = (N % 256 == 0) ? 256 : 128;
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_GROUPED;
  p.epi = mx::EPI_BF16;
  p.G = G;
  p.offsets = offsets_dev;
  p.R = R; p.K = K; p.Nb = N;
  p.a_type = mma_type(a->fmt); p.b_type = mma_type(b->fmt);
  p.sfa = a->scale; p.sfb = b->scale;
  p.sfa_kchunks = (K / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  p.m_tiles = (int)((R + 127) / 128);
  p.n_tiles = (int)(N / bn);
  p.num_tiles = (int64_t)p.m_tiles * p.n_tiles;
  p.out = static_cast<uint16_t*>(out_bf16);
  p.out_ld = ld_out;
  p.bias = static_cast<const uint16_t*>(bias_bf16);
  p.bias_ld = N;
  return run_gemm(p, a, b, bn, s, dev, OutView{out_bf16, R, N, ld_out});
}

}  // namespace

namespace {
mx_status_t pair_gemm_impl(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                           const void* bias_bf16, int64_t bias_ld, void* out_bf16, int64_t ld_out,
                           mx_stream_t stream);
}  // namespace

extern "C" {

mx_status_t mx_grouped_gemm(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                            void* out_bf16, int64_t ld_out, mx_stream_t stream) {
  return grouped_gemm_impl(a, b, G, offsets_dev, nullptr, out_bf16, ld_out, stream);
}

mx_status_t mx_grouped_gemm_2sm(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                                void* out_bf16, int64_t ld_out, mx_stream_t stream) {
  return pair_gemm_impl(a, b, G, offsets_dev, nullptr, 0, out_bf16, ld_out, stream);
}

}  // extern "C"

namespace {

// The CTA-pair grouped GEMM with an optional BF16 bias ([G, N] rows bias_ld
// apart, or one row of N with bias_ld 0) added before the single rounding.
mx_status_t pair_gemm_impl(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                           const void* bias_bf16, int64_t bias_ld, void* out_bf16, int64_t ld_out,
                           mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(a, "a")) != MX_OK) return st;
  if ((st = check_gemm_operand(b, "b")) != MX_OK) return st;
  if ((st = check_pair(a, b, "a", "b")) != MX_OK) return st;
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  MX_CHECK(a->cols == b->cols, MX_ERR_SHAPE, "a has K = %lld, b has K = %lld", (long long)a->cols, (long long)b->cols);
  const int64_t K = a->cols, R = a->rows;
  MX_CHECK(K % 128 == 0, MX_ERR_SHAPE, "K = %lld is not a multiple of 128", (long long)K);
  MX_CHECK(b->rows % G == 0, MX_ERR_SHAPE, "b has %lld rows, not a multiple of G = %d", (long long)b->rows, G);
  const int64_t N = b->rows / G;
  MX_CHECK(N > 0 && N % 256 == 0, MX_ERR_SHAPE, "N = %lld per expert is not a positive multiple of 256",
           (long long)N);
  MX_CHECK(R % 128 == 0, MX_ERR_SHAPE, "R = %lld is not a multiple of 128", (long long)R);
  MX_CHECK(G <= 1024, MX_ERR_NOT_SUPPORTED, "G = %d; the CTA-pair GEMM takes at most 1024 experts", G);
  MX_CHECK(R == 0 || (out_bf16 != nullptr && aligned16(out_bf16)), MX_ERR_ALIGNMENT,
           "out must be a 16-byte aligned pointer");
  MX_CHECK(ld_out >= N && ld_out % 8 == 0, MX_ERR_ALIGNMENT, "ld_out = %lld must be >= N and a multiple of 8",
           (long long)ld_out);
  MX_CHECK(R * ld_out < (1ll << 40), MX_ERR_SHAPE, "output too large");
  if ((st = check_offsets(offsets_dev, G, R, s)) != MX_OK) return st;
  if (R == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::PairParams p;
  memset(&p, 0, sizeof(p));
  MX_CHECK(bias_bf16 == nullptr || aligned16(bias_bf16), MX_ERR_ALIGNMENT, "bias must be a 16-byte aligned pointer");
  p.G = G; p.offsets = offsets_dev;
  p.R = R; p.K = K; p.Nb = N;
  p.a_type = mma_type(a->fmt); p.b_type = mma_type(b->fmt);
  p.bias = static_cast<const uint16_t*>(bias_bf16);
  p.bias_ld = bias_ld;
  p.n_tiles = N / 256;
  // 256-row tiles per expert segment: at most R / 256 plus one half-filled
  // tile for every expert with an odd number of 128-row blocks
  p.num_tiles = ((R + 255) / 256 + (offsets_dev ? (G + 1) / 2 : 0)) * p.n_tiles;
  // E2M1 runs on .kind::mxf4 from the packed payload: a stage is 128 bytes
  // (256 elements) of each row and two scale chunks, every box counted whole
  // (past K it is zero-filled).
  p.f4 = a->fmt == MX_E2M1 ? 1 : 0;
  const int kc = p.f4 ? 2 : 1;
  // one CTA's stage: 128 A rows, 128 B rows, A's chunks and both B row blocks' chunks
  p.tx_bytes = p.f4 ? 2u * 16384u + 3u * 1024u : stage_tx_bytes(a->fmt, 128) + 512u;
  CUtensorMap ta, tb, tsa, tsb, to;
  if ((st = p.f4 ? make_tmap_packed(&ta, a->data, a->rows, a->cols)
                 : make_tmap(&ta, a->data, a->rows, a->cols, a->fmt)) != MX_OK)
    return st;
  if ((st = p.f4 ? make_tmap_packed(&tb, b->data, b->rows, b->cols)
                 : make_tmap(&tb, b->data, b->rows, b->cols, b->fmt)) != MX_OK)
    return st;
  if ((st = make_tmap_scales(&tsa, a->scale, a->rows, K, 1, kc)) != MX_OK) return st;
  if ((st = make_tmap_scales(&tsb, b->scale, b->rows, K, 2, kc)) != MX_OK) return st;
  if ((st = make_tmap_out(&to, out_bf16, R, N, ld_out)) != MX_OK) return st;
  log_config("gemm pair bf16 BN=256%s a=%d b=%d R=%lld K=%lld N=%lld G=%d tiles=%lld", p.f4 ? " mxf4" : "",
             p.a_type, p.b_type, (long long)R, (long long)K, (long long)N, G, (long long)p.num_tiles);
  cudaError_t e = mx::launch_gemm_pair(p, ta, tb, tsa, tsb, to, s, dev.sms);
  if (e != cudaSuccess) return cuda_fail(e, "CTA-pair GEMM launch");
  return MX_OK;
}

}  // namespace

extern "C" {

mx_status_t mx_grouped_gemm_bias(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets_dev,
                                 const void* bias_bf16, void* out_bf16, int64_t ld_out, mx_stream_t stream) {
  MX_CHECK(bias_bf16 != nullptr && aligned16(bias_bf16), MX_ERR_ALIGNMENT, "bias must be a 16-byte aligned pointer");
  return grouped_gemm_impl(a, b, G, offsets_dev, bias_bf16, out_bf16, ld_out, stream);
}

mx_status_t mx_grouped_gemm_bias_2sm(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G,
                                     const int32_t* offsets_dev, const void* bias_bf16, void* out_bf16,
                                     int64_t ld_out, mx_stream_t stream) {
  MX_CHECK(bias_bf16 != nullptr && aligned16(bias_bf16), MX_ERR_ALIGNMENT, "bias must be a 16-byte aligned pointer");
  MX_CHECK(a != nullptr && b != nullptr && G >= 1, MX_ERR_INVALID_ARG, "a, b and G >= 1 are required");
  return pair_gemm_impl(a, b, G, offsets_dev, bias_bf16, b->rows / G, out_bf16, ld_out, stream);
}

}  // extern "C"

namespace {

mx_status_t swiglu_fwd_impl(const mx_tensor_t* x_row, const mx_tensor_t* w1_row, int32_t G,
                            const int32_t* offsets_dev, const float* probs, const mx_tensor_t* h_row,
                            const mx_tensor_t* h_col, void* z_bf16, mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(x_row, "x_row")) != MX_OK) return st;
  if ((st = check_gemm_operand(w1_row, "w1_row")) != MX_OK) return st;
  if ((st = check_pair(x_row, w1_row, "x_row", "w1_row")) != MX_OK) return st;
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  const int64_t R = x_row->rows, D = x_row->cols;
  MX_CHECK(w1_row->cols == D, MX_ERR_SHAPE, "w1_row has K = %lld, x_row has %lld", (long long)w1_row->cols,
           (long long)D);
  MX_CHECK(D % 128 == 0, MX_ERR_SHAPE, "D = %lld is not a multiple of 128", (long long)D);
  MX_CHECK(R % 128 == 0, MX_ERR_SHAPE, "R = %lld is not a multiple of 128", (long long)R);
  MX_CHECK(w1_row->rows % (2ll * G) == 0, MX_ERR_SHAPE, "w1_row rows %lld is not 2F*G", (long long)w1_row->rows);
  const int64_t F = w1_row->rows / (2ll * G);
  MX_CHECK(F > 0 && F % 128 == 0, MX_ERR_SHAPE, "F = %lld is not a positive multiple of 128", (long long)F);
  if ((st = check_tensor(h_row, "h_row", R, F, MX_E4M3, 0)) != MX_OK) return st;
  if ((st = check_tensor(h_col, "h_col", F, R, MX_E4M3, 0)) != MX_OK) return st;
  MX_CHECK(z_bf16 != nullptr && aligned16(z_bf16), MX_ERR_ALIGNMENT, "z must be a 16-byte aligned pointer");
  MX_CHECK(R * 2 * F < (1ll << 40), MX_ERR_SHAPE, "output too large");
  if ((st = check_offsets(offsets_dev, G, R, s)) != MX_OK) return st;
  if (R == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_GROUPED;
  p.epi = mx::EPI_SWIGLU;
  p.G = G; p.offsets = offsets_dev;
  p.R = R; p.K = D; p.Nb = 2 * F; p.F = F;
  p.a_type = mma_type(x_row->fmt); p.b_type = mma_type(w1_row->fmt);
  p.sfa = x_row->scale; p.sfb = w1_row->scale;
  p.sfa_kchunks = (D / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  p.m_tiles = (int)(R / 128);
  p.n_tiles = (int)(F / 128);
  p.num_tiles = (int64_t)p.m_tiles * p.n_tiles;
  p.z = static_cast<uint16_t*>(z_bf16);
  p.probs = probs;
  p.q_row = static_cast<uint8_t*>(h_row->data); p.q_row_scale = h_row->scale;
  p.q_col = static_cast<uint8_t*>(h_col->data); p.q_col_scale = h_col->scale;
  p.q_cols = F;
  if ((st = attach_tap(&p, R, F)) != MX_OK) return st;
  return run_gemm(p, x_row, w1_row, 256, s, dev, OutView{z_bf16, R, 2 * F, 2 * F},
                  fused_pairs_enabled(true) && G <= mx::MAX_PAIR_G_HOST);
}

}  // namespace

extern "C" {

mx_status_t mx_grouped_gemm_swiglu_fwd(const mx_tensor_t* x_row, const mx_tensor_t* w1_row, int32_t G,
                                       const int32_t* offsets_dev, const mx_tensor_t* h_row,
                                       const mx_tensor_t* h_col, void* z_bf16, mx_stream_t stream) {
  return swiglu_fwd_impl(x_row, w1_row, G, offsets_dev, nullptr, h_row, h_col, z_bf16, stream);
}

mx_status_t mx_grouped_gemm_swiglu_probs_fwd(const mx_tensor_t* x_row, const mx_tensor_t* w1_row, int32_t G,
                                             const int32_t* offsets_dev, const float* probs,
                                             const mx_tensor_t* h_row, const mx_tensor_t* h_col, void* z_bf16,
                                             mx_stream_t stream) {
  MX_CHECK(probs != nullptr && aligned16(probs), MX_ERR_ALIGNMENT, "probs must be a 16-byte aligned pointer");
  return swiglu_fwd_impl(x_row, w1_row, G, offsets_dev, probs, h_row, h_col, z_bf16, stream);
}

}  // extern "C"

namespace {

mx_status_t dswiglu_bwd_impl(const mx_tensor_t* dy_row, const mx_tensor_t* w2t_row, const void* z_bf16,
                             const float* probs, int32_t G, const int32_t* offsets_dev, const mx_tensor_t* dz_row,
                             const mx_tensor_t* dz_col, float* dprobs, void* workspace, size_t workspace_bytes,
                             mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(dy_row, "dy_row")) != MX_OK) return st;
  if ((st = check_gemm_operand(w2t_row, "w2t_row")) != MX_OK) return st;
  if ((st = check_pair(dy_row, w2t_row, "dy_row", "w2t_row")) != MX_OK) return st;
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  const int64_t R = dy_row->rows, D = dy_row->cols;
  MX_CHECK(w2t_row->cols == D, MX_ERR_SHAPE, "w2t_row has K = %lld, dy_row has %lld", (long long)w2t_row->cols,
           (long long)D);
  MX_CHECK(D % 128 == 0, MX_ERR_SHAPE, "D = %lld is not a multiple of 128", (long long)D);
  MX_CHECK(R % 128 == 0, MX_ERR_SHAPE, "R = %lld is not a multiple of 128", (long long)R);
  MX_CHECK(w2t_row->rows % G == 0, MX_ERR_SHAPE, "w2t_row rows %lld is not F*G", (long long)w2t_row->rows);
  const int64_t F = w2t_row->rows / G;
  MX_CHECK(F > 0 && F % 128 == 0, MX_ERR_SHAPE, "F = %lld is not a positive multiple of 128", (long long)F);
  if ((st = check_tensor(dz_row, "dz_row", R, 2 * F, MX_E4M3, 0)) != MX_OK) return st;
  if ((st = check_tensor(dz_col, "dz_col", 2 * F, R, MX_E4M3, 0)) != MX_OK) return st;
  MX_CHECK(z_bf16 != nullptr && aligned16(z_bf16), MX_ERR_ALIGNMENT, "z must be a 16-byte aligned pointer");
  MX_CHECK(R * 2 * F < (1ll << 40), MX_ERR_SHAPE, "output too large");
  if ((st = check_offsets(offsets_dev, G, R, s)) != MX_OK) return st;
  if (R == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_GROUPED;
  p.epi = mx::EPI_DSWIGLU;
  p.G = G; p.offsets = offsets_dev;
  p.R = R; p.K = D; p.Nb = F; p.F = F;
  p.a_type = mma_type(dy_row->fmt); p.b_type = mma_type(w2t_row->fmt);
  p.sfa = dy_row->scale; p.sfb = w2t_row->scale;
  p.sfa_kchunks = (D / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  // 256-column tiles (the 128x256 MMA) where F allows, else 128
  const int tile_n = F % 256 == 0 ? 256 : 128;
  const bool pair = tile_n == 256 && fused_pairs_enabled(false) && G <= mx::MAX_PAIR_G_HOST;
  p.m_tiles = (int)(R / 128);
  p.n_tiles = (int)(F / tile_n);
  p.num_tiles = (int64_t)p.m_tiles * p.n_tiles;
  p.z = static_cast<uint16_t*>(const_cast<void*>(z_bf16));
  p.q_row = static_cast<uint8_t*>(dz_row->data); p.q_row_scale = dz_row->scale;
  p.q_col = static_cast<uint8_t*>(dz_col->data); p.q_col_scale = dz_col->scale;
  p.q_cols = 2 * F;
  if ((st = attach_tap(&p, R, 2 * F)) != MX_OK) return st;
  if (probs != nullptr) {
    const int64_t ld = 2 * (F / tile_n);  // one partial per tile and column half
    MX_CHECK(dprobs != nullptr, MX_ERR_INVALID_ARG, "dprobs is NULL");
    MX_CHECK(workspace != nullptr && aligned16(workspace) && workspace_bytes >= (size_t)(R * ld * 4),
             MX_ERR_WORKSPACE, "the probabilities' workspace needs %lld bytes", (long long)(R * ld * 4));
    p.probs = probs;
    p.dprobs_part = static_cast<float*>(workspace);
    p.dprobs_ld = ld;
    if ((st = run_gemm(p, dy_row, w2t_row, tile_n, s, dev, OutView{nullptr, 0, 0, 0}, pair)) != MX_OK) return st;
    cudaError_t e = mx::launch_dprobs_reduce(p.dprobs_part, R, ld, offsets_dev, G, dprobs, s);
    if (e != cudaSuccess) return cuda_fail(e, "dprobs reduction launch");
    return MX_OK;
  }
  return run_gemm(p, dy_row, w2t_row, tile_n, s, dev, OutView{nullptr, 0, 0, 0}, pair);
}

}  // namespace

extern "C" {

mx_status_t mx_grouped_gemm_dswiglu_bwd(const mx_tensor_t* dy_row, const mx_tensor_t* w2t_row, const void* z_bf16,
                                        int32_t G, const int32_t* offsets_dev, const mx_tensor_t* dz_row,
                                        const mx_tensor_t* dz_col, mx_stream_t stream) {
  return dswiglu_bwd_impl(dy_row, w2t_row, z_bf16, nullptr, G, offsets_dev, dz_row, dz_col, nullptr, nullptr, 0,
                          stream);
}

size_t mx_dswiglu_probs_workspace_bytes(int64_t R, int64_t F) {
  if (R < 0 || F <= 0) return 0;
  return (size_t)R * (size_t)(2 * ((F + 127) / 128)) * 4;
}

mx_status_t mx_grouped_gemm_dswiglu_probs_bwd(const mx_tensor_t* dy_row, const mx_tensor_t* w2t_row,
                                              const void* z_bf16, const float* probs, int32_t G,
                                              const int32_t* offsets_dev, const mx_tensor_t* dz_row,
                                              const mx_tensor_t* dz_col, float* dprobs, void* workspace,
                                              size_t workspace_bytes, mx_stream_t stream) {
  MX_CHECK(probs != nullptr && aligned16(probs), MX_ERR_ALIGNMENT, "probs must be a 16-byte aligned pointer");
  MX_CHECK(dprobs != nullptr && aligned16(dprobs), MX_ERR_ALIGNMENT, "dprobs must be a 16-byte aligned pointer");
  return dswiglu_bwd_impl(dy_row, w2t_row, z_bf16, probs, G, offsets_dev, dz_row, dz_col, dprobs, workspace,
                          workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Ragged-K wgrad into BF16 (EPI_BF16) or into an fp32 gradient buffer
// (EPI_F32, stored or accumulated).
// Wgrad K-split geometry for N output rows, K output columns and R routed
// rows: tiles per expert, when an expert is split (more 128-row chunks than
// `trigger`: one of its tiles would run longer than half the average work
// per SM) and into parts of how many chunks (`chunks`, a quarter of that
// work), and the workspace (arrival counters, then fp32 partial tiles).
// Measured at 262144 routed rows under Zipf(1.1) routing: parts of 1/4 of
// the per-SM work cut dW2 (48 tiles per expert) from 465 to 407 us; parts of
// 1/8 and 1/16 were slower than no split (the partial tiles' traffic), and
// dW1 (96 tiles per expert) gains nothing, which the trigger leaves alone.
struct WgradSplit {
  int bn;
  int64_t per_g, chunks, trigger, slots, extra;
  size_t cnt_bytes, bytes;
};

WgradSplit wgrad_split(int64_t N, int64_t K, int64_t R, int num_sms) {
  WgradSplit w;
  w.bn = (K % 256 == 0) ? 256 : 128;
  w.per_g = (N / 128) * (K / w.bn);
  const int64_t total = R / 128;
  const int64_t per_sm = total * w.per_g / (num_sms > 0 ? num_sms : 148);
  w.trigger = per_sm / 2 < 64 ? 64 : per_sm / 2;
  const int64_t c = per_sm / 4;
  w.chunks = c < 64 ? 64 : (c > 4096 ? 4096 : c);
  w.extra = w.per_g * (total / w.chunks);
  w.slots = w.per_g * (2 * total / w.chunks);
  // the split parts' arrival counters, then the dynamic schedule's tile counter
  w.cnt_bytes = align_up(((size_t)mx::MAX_SPLIT_EXPERTS * (size_t)w.per_g + 1) * 4);
  w.bytes = w.slots > 0 ? w.cnt_bytes + (size_t)w.slots * 128 * (size_t)w.bn * 4 : 0;
  return w;
}

mx_status_t wgrad_common(const mx_tensor_t* a_col, const mx_tensor_t* b_col, int32_t G, const int32_t* offsets_dev,
                         void* out, int epi, int accumulate, void* workspace, size_t workspace_bytes,
                         mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(a_col, "a_col")) != MX_OK) return st;
  if ((st = check_gemm_operand(b_col, "b_col")) != MX_OK) return st;
  if ((st = check_pair(a_col, b_col, "a_col", "b_col")) != MX_OK) return st;
  MX_CHECK(G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", G);
  const int64_t N = a_col->rows, K = b_col->rows, R = a_col->cols;
  MX_CHECK(b_col->cols == R, MX_ERR_SHAPE, "a_col has R = %lld, b_col has %lld", (long long)R,
           (long long)b_col->cols);
  MX_CHECK(R % 128 == 0, MX_ERR_SHAPE, "R = %lld is not a multiple of 128", (long long)R);
  MX_CHECK(N > 0 && N % 128 == 0, MX_ERR_SHAPE, "N = %lld is not a positive multiple of 128", (long long)N);
  MX_CHECK(K > 0 && K % 128 == 0, MX_ERR_SHAPE, "K = %lld is not a positive multiple of 128", (long long)K);
  MX_CHECK(out != nullptr && aligned16(out), MX_ERR_ALIGNMENT, "out must be a 16-byte aligned pointer");
  MX_CHECK((int64_t)G * N * K < (1ll << 40), MX_ERR_SHAPE, "output too large");
  if ((st = check_offsets(offsets_dev, G, R, s)) != MX_OK) return st;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  const int bn = (K % 256 == 0) ? 256 : 128;
  // CTA pairs on 256 x 256 tiles where the weight's rows and columns allow
  const bool pair = bn == 256 && N % 256 == 0 && a_col->fmt != MX_E2M1 && fused_pairs_enabled(false);
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_WGRAD;
  p.epi = epi;
  p.G = G; p.offsets = offsets_dev;
  p.R = R; p.K = R; p.Nb = K; p.Mw = N;
  p.a_type = mma_type(a_col->fmt); p.b_type = mma_type(b_col->fmt);
  p.sfa = a_col->scale; p.sfb = b_col->scale;
  p.sfa_kchunks = (R / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  p.m_tiles = (int)(N / (pair ? 256 : 128));
  p.n_tiles = (int)(K / bn);
  p.num_tiles = (int64_t)G * p.m_tiles * p.n_tiles;
  if (epi == mx::EPI_F32) {
    p.out_f32 = static_cast<float*>(out);
    p.accumulate = accumulate ? 1 : 0;
  } else {
    p.out = static_cast<uint16_t*>(out);
  }
  p.out_ld = K;
  // K-split of the largest experts when a workspace is given (and there is
  // a ranking: offsets, 1 < G <= 1024)
  const WgradSplit w = wgrad_split(N, K, R, dev.sms);
  if (workspace != nullptr && w.bytes > 0 && offsets_dev != nullptr && G > 1 && G <= 1024) {
    MX_CHECK(aligned16(workspace) && workspace_bytes >= w.bytes, MX_ERR_WORKSPACE,
             "the split wgrad needs %zu bytes of 16-byte aligned workspace (mx_grouped_gemm_wgrad_workspace_bytes)",
             w.bytes);
    p.split_chunks = (int)w.chunks;
    p.split_min = (int)w.trigger;
    p.split_cnt = static_cast<int32_t*>(workspace);
    p.dyn_ctr = p.split_cnt + (int64_t)mx::MAX_SPLIT_EXPERTS * w.per_g;
    p.split_ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.cnt_bytes);
    p.split_slots = w.slots;
    // pairs: the extra tiles (and the kernel's slots) count 256-row tiles,
    // half as many; the workspace's slots and counters are the same bytes
    p.split_extra = pair ? w.extra / 2 : w.extra;
    p.num_tiles += p.split_extra;
    cudaError_t e = cudaMemsetAsync(workspace, 0, w.cnt_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the split counters");
  }
  return run_gemm(p, a_col, b_col, bn, s, dev, OutView{out, (int64_t)G * N, K, K, epi == mx::EPI_F32}, pair);
}

}  // namespace

extern "C" {

mx_status_t mx_grouped_gemm_wgrad(const mx_tensor_t* a_col, const mx_tensor_t* b_col, int32_t G,
                                  const int32_t* offsets_dev, void* out_bf16, mx_stream_t stream) {
  return wgrad_common(a_col, b_col, G, offsets_dev, out_bf16, mx::EPI_BF16, 0, nullptr, 0, stream);
}

mx_status_t mx_grouped_gemm_wgrad_f32(const mx_tensor_t* a_col, const mx_tensor_t* b_col, int32_t G,
                                      const int32_t* offsets_dev, float* grad_f32, int32_t accumulate,
                                      mx_stream_t stream) {
  MX_CHECK(accumulate == 0 || accumulate == 1, MX_ERR_INVALID_ARG, "accumulate = %d (0 stores, 1 adds)", accumulate);
  return wgrad_common(a_col, b_col, G, offsets_dev, grad_f32, mx::EPI_F32, accumulate, nullptr, 0, stream);
}

size_t mx_grouped_gemm_wgrad_workspace_bytes(int64_t N, int64_t K, int64_t R, int32_t G) {
  if (N <= 0 || K <= 0 || R <= 0 || G <= 1 || N % 128 || K % 128 || R % 128) return 0;
  DevInfo dev;
  const int sms = device_info(&dev) == MX_OK ? dev.sms : 0;
  return wgrad_split(N, K, R, sms).bytes;
}

mx_status_t mx_grouped_gemm_wgrad_ws(const mx_tensor_t* a_col, const mx_tensor_t* b_col, int32_t G,
                                     const int32_t* offsets_dev, void* out_bf16, void* workspace,
                                     size_t workspace_bytes, mx_stream_t stream) {
  return wgrad_common(a_col, b_col, G, offsets_dev, out_bf16, mx::EPI_BF16, 0, workspace, workspace_bytes, stream);
}

mx_status_t mx_grouped_gemm_wgrad_f32_ws(const mx_tensor_t* a_col, const mx_tensor_t* b_col, int32_t G,
                                         const int32_t* offsets_dev, float* grad_f32, int32_t accumulate,
                                         void* workspace, size_t workspace_bytes, mx_stream_t stream) {
  MX_CHECK(accumulate == 0 || accumulate == 1, MX_ERR_INVALID_ARG, "accumulate = %d (0 stores, 1 adds)", accumulate);
  return wgrad_common(a_col, b_col, G, offsets_dev, grad_f32, mx::EPI_F32, accumulate, workspace, workspace_bytes,
                      stream);
}


mx_status_t mx_gemm_bias(const mx_tensor_t* a, const mx_tensor_t* b, const void* bias_bf16, void* out_bf16,
                         int64_t ld_out, mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mx_status_t st;
  if ((st = check_gemm_operand(a, "a")) != MX_OK) return st;
  if ((st = check_gemm_operand(b, "b")) != MX_OK) return st;
  if ((st = check_pair(a, b, "a", "b")) != MX_OK) return st;
  const int64_t M = a->rows, K = a->cols, N = b->rows;
  MX_CHECK(b->cols == K, MX_ERR_SHAPE, "a has K = %lld, b has K = %lld", (long long)K, (long long)b->cols);
  MX_CHECK(K % 128 == 0 && M % 128 == 0 && N > 0 && N % 128 == 0, MX_ERR_SHAPE,
           "M = %lld, N = %lld, K = %lld must be multiples of 128", (long long)M, (long long)N, (long long)K);
  MX_CHECK(out_bf16 != nullptr && aligned16(out_bf16), MX_ERR_ALIGNMENT, "out must be a 16-byte aligned pointer");
  MX_CHECK(bias_bf16 == nullptr || aligned16(bias_bf16), MX_ERR_ALIGNMENT, "bias must be 16-byte aligned");
  MX_CHECK(ld_out >= N && ld_out % 8 == 0, MX_ERR_ALIGNMENT, "ld_out = %lld must be >= N and a multiple of 8",
           (long long)ld_out);
  if (M == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  const int bn = (N % 256 == 0) ? 256 : 128;
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_GROUPED;
  p.epi = mx::EPI_BF16;
  p.G = 1; p.offsets = nullptr;
  p.R = M; p.K = K; p.Nb = N;
  p.a_type = mma_type(a->fmt); p.b_type = mma_type(b->fmt);
  p.sfa = a->scale; p.sfb = b->scale;
  p.sfa_kchunks = (K / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  p.m_tiles = (int)(M / 128);
  p.n_tiles = (int)(N / bn);
  p.num_tiles = (int64_t)p.m_tiles * p.n_tiles;
  p.out = static_cast<uint16_t*>(out_bf16);
  p.out_ld = ld_out;
  p.bias = static_cast<const uint16_t*>(bias_bf16);
  return run_gemm(p, a, b, bn, s, dev, OutView{out_bf16, M, N, ld_out});
}

namespace {

// Shared set-up of the two dense fused epilogues: A [M, K], B [H, K],
// requant outputs q_row [M, H] and q_col [H, M] of one format and rotation.
mx_status_t dense_fused(int epi, const mx_tensor_t* a, const mx_tensor_t* b, const void* bias_bf16, void* pre_bf16,
                        const mx_tensor_t* q_row, const mx_tensor_t* q_col, float* partials, cudaStream_t s,
                        int64_t* M_out, int64_t* H_out) {
  mx_status_t st;
  const char* an = epi == mx::EPI_GELU ? "x_row" : "dy_row";
  const char* bn = epi == mx::EPI_GELU ? "w1_row" : "w2t_row";
  if ((st = check_gemm_operand(a, an)) != MX_OK) return st;
  if ((st = check_gemm_operand(b, bn)) != MX_OK) return st;
  if ((st = check_pair(a, b, an, bn)) != MX_OK) return st;
  const int64_t M = a->rows, K = a->cols, H = b->rows;
  *M_out = M;
  *H_out = H;
  MX_CHECK(b->cols == K, MX_ERR_SHAPE, "%s has K = %lld, %s has K = %lld", an, (long long)K, bn, (long long)b->cols);
  MX_CHECK(M % 128 == 0 && K % 128 == 0 && H > 0 && H % 128 == 0, MX_ERR_SHAPE,
           "M = %lld, H = %lld, K = %lld must be multiples of 128", (long long)M, (long long)H, (long long)K);
  MX_CHECK(q_row != nullptr && q_col != nullptr, MX_ERR_INVALID_ARG, "requant outputs are NULL");
  MX_CHECK(q_row->fmt == MX_E4M3 || q_row->fmt == MX_E2M3, MX_ERR_NOT_SUPPORTED,
           "the dense epilogues requantize to E4M3 or E2M3");
  if ((st = check_tensor(q_row, epi == mx::EPI_GELU ? "act_row" : "dpre_row", M, H, q_row->fmt, q_row->hadamard)) != MX_OK)
    return st;
  if ((st = check_tensor(q_col, epi == mx::EPI_GELU ? "act_col" : "dpre_col", H, M, q_row->fmt, q_row->hadamard)) != MX_OK)
    return st;
  MX_CHECK(pre_bf16 != nullptr && aligned16(pre_bf16), MX_ERR_ALIGNMENT, "pre must be a 16-byte aligned pointer");
  MX_CHECK(bias_bf16 == nullptr || aligned16(bias_bf16), MX_ERR_ALIGNMENT, "bias must be 16-byte aligned");
  if (M == 0) return MX_OK;
  DevInfo dev;
  if ((st = device_info(&dev)) != MX_OK) return st;
  mx::GemmParams p = base_params();
  p.mode = mx::MODE_GROUPED;
  p.epi = epi;
  p.G = 1; p.offsets = nullptr;
  p.R = M; p.K = K; p.Nb = H;
  p.a_type = mma_type(a->fmt); p.b_type = mma_type(b->fmt);
  p.sfa = a->scale; p.sfb = b->scale;
  p.sfa_kchunks = (K / 32 + 3) / 4;
  p.sfb_kchunks = p.sfa_kchunks;
  // 256-column tiles (the 128x256 MMA) where H allows, else 128
  const int tile_n = H % 256 == 0 ? 256 : 128;
  p.m_tiles = (int)(M / 128);
  p.n_tiles = (int)(H / tile_n);
  p.num_tiles = (int64_t)p.m_tiles * p.n_tiles;
  p.z = static_cast<uint16_t*>(pre_bf16);
  p.q_row = static_cast<uint8_t*>(q_row->data); p.q_row_scale = q_row->scale;
  p.q_col = static_cast<uint8_t*>(q_col->data); p.q_col_scale = q_col->scale;
  p.q_cols = H;
  p.q_row_ld = mx::payload_row_bytes(H, q_row->fmt);
  p.q_col_ld = mx::payload_row_bytes(M, q_row->fmt);
  p.q_fmt = q_row->fmt;
  p.q_had = q_row->hadamard ? 1 : 0;
  p.bias = static_cast<const uint16_t*>(bias_bf16);
  p.colsum_partials = partials;
  p.tx_bytes = stage_tx_bytes(a->fmt, tile_n);
  CUtensorMap ta, tb, to;
  if ((st = make_tmap(&ta, a->data, a->rows, a->cols, a->fmt)) != MX_OK) return st;
  if ((st = make_tmap(&tb, b->data, b->rows, b->cols, b->fmt)) != MX_OK) return st;
  if (epi == mx::EPI_GELU) {
    if ((st = make_tmap_out(&to, pre_bf16, M, H, H)) != MX_OK) return st;
  } else {
    to = ta;
  }
  if ((st = attach_tap(&p, p.R, p.q_cols)) != MX_OK) return st;
  log_config("gemm dense %s BN=%d a=%d out_fmt=%d rotated=%d M=%lld K=%lld N=%lld tiles=%lld grid=%lld",
             epi_name(p.epi), tile_n, p.a_type, p.q_fmt, p.q_had, (long long)p.R, (long long)p.K, (long long)p.Nb,
             (long long)p.num_tiles, (long long)(p.num_tiles < dev.sms ? p.num_tiles : dev.sms));
  cudaError_t e = mx::launch_gemm_dense(p, ta, tb, to, tile_n, s, dev.sms);
  if (e != cudaSuccess) return cuda_fail(e, "dense GEMM launch");
  return MX_OK;
}

}  // namespace

mx_status_t mx_gemm_gelu_fwd(const mx_tensor_t* x_row, const mx_tensor_t* w1_row, const void* b1_bf16,
                             void* pre_bf16, const mx_tensor_t* act_row, const mx_tensor_t* act_col,
                             mx_stream_t stream) {
  int64_t M, H;
  return dense_fused(mx::EPI_GELU, x_row, w1_row, b1_bf16, pre_bf16, act_row, act_col, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), &M, &H);
}

size_t mx_gemm_dgelu_workspace_bytes(int64_t M, int64_t H) {
  if (M <= 0 || H <= 0) return 0;
  return (size_t)((M + 127) / 128) * (size_t)H * sizeof(float);
}

mx_status_t mx_gemm_dgelu_bwd(const mx_tensor_t* dy_row, const mx_tensor_t* w2t_row, const void* pre_bf16,
                              const mx_tensor_t* dpre_row, const mx_tensor_t* dpre_col, float* db1, void* workspace,
                              size_t workspace_bytes, mx_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MX_CHECK(dy_row != nullptr && w2t_row != nullptr, MX_ERR_INVALID_ARG, "operands are NULL");
  const int64_t M0 = dy_row->rows, H0 = w2t_row->rows;
  MX_CHECK(db1 != nullptr && aligned16(db1), MX_ERR_INVALID_ARG, "db1 must be a 16-byte aligned pointer");
  MX_CHECK(workspace != nullptr && aligned16(workspace) && workspace_bytes >= mx_gemm_dgelu_workspace_bytes(M0, H0),
           MX_ERR_WORKSPACE, "needs %zu bytes of 16-byte aligned workspace", mx_gemm_dgelu_workspace_bytes(M0, H0));
  int64_t M, H;
  mx_status_t st = dense_fused(mx::EPI_DGELU, dy_row, w2t_row, nullptr, const_cast<void*>(pre_bf16), dpre_row,
                               dpre_col, static_cast<float*>(workspace), s, &M, &H);
  if (st != MX_OK || M == 0) return st;
  cudaError_t e = mx::launch_colsum_reduce(static_cast<const float*>(workspace), M / 128, H, db1, s);
  if (e != cudaSuccess) return cuda_fail(e, "column-sum reduce launch");
  return MX_OK;
}

// ---- the MLP step -------------------------------------------------------

namespace {

// Workspace of one MLP step: every quantized operand between the stages,
// the BF16 pre-activation and (GELU) the column-sum partials.
struct MlpLayout {
  size_t total = 0;
  struct Slot { size_t data, scale; int64_t rows, cols; };
  Slot x_row, x_col, w1_row, w1t_row, w2_row, w2t_row, h_row, h_col, dy_row, dy_col, dz_row, dz_col;
  size_t z, part_dy, part_dz;
  size_t split, split_bytes;  // wgrad K-split workspace (0 bytes: no split)
};


MlpLayout mlp_layout(const mx_mlp_args_t* a) {
  MlpLayout L;
  size_t off = 0;
  const int fmt = a->fmt;
  auto slot = [&](int64_t rows, int64_t cols) {
    MlpLayout::Slot s;
    s.rows = rows; s.cols = cols;
    s.data = off; off = align_up(off + (size_t)rows * (size_t)mx::payload_row_bytes(cols, fmt));
    s.scale = off; off = align_up(off + mx::scale_bytes(rows, cols / 32));
    return s;
  };
  const int64_t R = a->R, D = a->D, F = a->F, G = a->G;
  const bool glu = a->act == MX_ACT_SWIGLU;
  const int64_t F1 = glu ? 2 * F : F;  // FC1 output width
  L.x_row = slot(R, D);
  L.x_col = slot(D, R);
  L.w1_row = slot(G * F1, D);
  L.w1t_row = slot(G * D, F1);
  L.w2_row = slot(G * D, F);
  L.w2t_row = slot(G * F, D);
  L.h_row = slot(R, F);
  L.h_col = slot(F, R);
  L.dy_row = slot(R, D);
  L.dy_col = slot(D, R);
  L.dz_row = slot(R, F1);
  L.dz_col = slot(F1, R);
  L.z = off; off = align_up(off + (size_t)R * (size_t)F1 * 2);
  L.part_dy = L.part_dz = off;
  if (!glu) {
    L.part_dy = off; off = align_up(off + (size_t)((R + 127) / 128) * (size_t)D * 4);
    L.part_dz = off; off = align_up(off + (size_t)((R + 127) / 128) * (size_t)F * 4);
  }
  L.split = off;
  L.split_bytes = 0;
  if (glu && G > 1) {
    DevInfo dev;
    const int sms = device_info(&dev) == MX_OK ? dev.sms : 0;
    const size_t b2 = wgrad_split(D, F, R, sms).bytes, b1 = wgrad_split(F1, D, R, sms).bytes;
    L.split_bytes = b1 > b2 ? b1 : b2;
    off = align_up(off + L.split_bytes);
  }
  L.total = off;
  return L;
}

mx_tensor_t view(const mx_mlp_args_t* a, const MlpLayout::Slot& s) {
  mx_tensor_t t;
  uint8_t* base = static_cast<uint8_t*>(a->workspace);
  t.data = base + s.data;
  t.scale = base + s.scale;
  t.rows = s.rows; t.cols = s.cols;
  t.fmt = a->fmt; t.hadamard = a->hadamard ? 1 : 0;
  return t;
}

// Stage hooks (the host pipeline orders its copies against these points;
// without hooks the step is the plain chain).
struct HookCall {
  const mx::StepHooks* h;
  void pre(int t) const { if (h) h->before(h->ctx, t); }
  void post(int t) const { if (h) h->after(h->ctx, t); }
};

// The step's plain grouped GEMMs (FC2, FC1 dgrad): on CTA pairs when the
// output width is a multiple of 256 (3-13 % faster than one SM per tile),
// else on the single-SM kernel; the outputs are the same bit for bit.
mx_status_t plain_gemm(const mx_tensor_t* a, const mx_tensor_t* b, int32_t G, const int32_t* offsets, void* out,
                       int64_t ld, mx_stream_t stream) {
  const int64_t N = G > 0 ? b->rows / G : 0;
  if (N > 0 && N % 256 == 0 && G <= 1024) return mx_grouped_gemm_2sm(a, b, G, offsets, out, ld, stream);
  return mx_grouped_gemm(a, b, G, offsets, out, ld, stream);
}

mx_status_t mlp_swiglu(const mx_mlp_args_t* a, const MlpLayout& L, mx_stream_t stream, const mx::StepHooks* hooks) {
  const int64_t R = a->R, D = a->D, F = a->F, G = a->G;
  mx_tensor_t x_row = view(a, L.x_row), x_col = view(a, L.x_col);
  mx_tensor_t w1_row = view(a, L.w1_row), w1t_row = view(a, L.w1t_row);
  mx_tensor_t w2_row = view(a, L.w2_row), w2t_row = view(a, L.w2t_row);
  mx_tensor_t h_row = view(a, L.h_row), h_col = view(a, L.h_col);
  mx_tensor_t dy_row = view(a, L.dy_row), dy_col = view(a, L.dy_col);
  mx_tensor_t dz_row = view(a, L.dz_row), dz_col = view(a, L.dz_col);
  void* z = static_cast<uint8_t*>(a->workspace) + L.z;
  const uint32_t both = MX_ROWWISE | MX_COLWISE;
  const HookCall hk{hooks};
  mx_status_t st;
  hk.pre(mx::T_X);
  if ((st = mx_quantize(a->x, 1, R, D, D, MX_E4M3, both, &x_row, &x_col, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_X);
  hk.pre(mx::T_W1);
  if ((st = mx_quantize(a->w1, G, 2 * F, D, D, MX_E4M3, both, &w1_row, &w1t_row, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_W1);
  hk.pre(mx::T_W2);
  if ((st = mx_quantize(a->w2, G, D, F, F, MX_E4M3, both, &w2_row, &w2t_row, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_W2);
  if ((st = mx_grouped_gemm_swiglu_fwd(&x_row, &w1_row, a->G, a->offsets, &h_row, &h_col, z, stream)) != MX_OK) return st;
  hk.pre(mx::T_Y);
  if ((st = plain_gemm(&h_row, &w2_row, a->G, a->offsets, a->y, D, stream)) != MX_OK) return st;
  hk.post(mx::T_Y);
  hk.pre(mx::T_DY);
  if ((st = mx_quantize(a->dy, 1, R, D, D, MX_E4M3, both, &dy_row, &dy_col, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_DY);
  if ((st = mx_grouped_gemm_dswiglu_bwd(&dy_row, &w2t_row, z, a->G, a->offsets, &dz_row, &dz_col, stream)) != MX_OK) return st;
  hk.pre(mx::T_DX);
  if ((st = plain_gemm(&dz_row, &w1t_row, a->G, a->offsets, a->dx, D, stream)) != MX_OK) return st;
  hk.post(mx::T_DX);
  hk.pre(mx::T_DW2);
  void* split_ws = L.split_bytes ? static_cast<uint8_t*>(a->workspace) + L.split : nullptr;
  if ((st = mx_grouped_gemm_wgrad_ws(&dy_col, &h_col, a->G, a->offsets, a->dw2, split_ws, L.split_bytes, stream)) !=
      MX_OK)
    return st;
  hk.post(mx::T_DW2);
  hk.pre(mx::T_DW1);
  if ((st = mx_grouped_gemm_wgrad_ws(&dz_col, &x_col, a->G, a->offsets, a->dw1, split_ws, L.split_bytes, stream)) !=
      MX_OK)
    return st;
  hk.post(mx::T_DW1);
  return MX_OK;
}

// Dense GELU step ([MXFP6-PR] fused-MLP commit): 12 launches.
mx_status_t mlp_gelu(const mx_mlp_args_t* a, const MlpLayout& L, mx_stream_t stream, const mx::StepHooks* hooks) {
  const int64_t M = a->R, D = a->D, H = a->F;
  const int fmt = a->fmt;
  const uint32_t both = MX_ROWWISE | MX_COLWISE | (a->hadamard ? MX_HADAMARD : 0);
  mx_tensor_t x_row = view(a, L.x_row), x_col = view(a, L.x_col);
  mx_tensor_t w1_row = view(a, L.w1_row), w1t_row = view(a, L.w1t_row);
  mx_tensor_t w2_row = view(a, L.w2_row), w2t_row = view(a, L.w2t_row);
  mx_tensor_t act_row = view(a, L.h_row), act_col = view(a, L.h_col);
  mx_tensor_t dy_row = view(a, L.dy_row), dy_col = view(a, L.dy_col);
  mx_tensor_t dpre_row = view(a, L.dz_row), dpre_col = view(a, L.dz_col);
  uint8_t* base = static_cast<uint8_t*>(a->workspace);
  void* pre = base + L.z;
  const size_t part_dy_bytes = (size_t)((M + 127) / 128) * (size_t)D * 4;
  const size_t part_dz_bytes = (size_t)((M + 127) / 128) * (size_t)H * 4;
  const HookCall hk{hooks};
  mx_status_t st;
  hk.pre(mx::T_X);
  if ((st = mx_quantize(a->x, 1, M, D, D, fmt, both, &x_row, &x_col, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_X);
  hk.pre(mx::T_W1);
  if ((st = mx_quantize(a->w1, 1, H, D, D, fmt, both, &w1_row, &w1t_row, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_W1);
  hk.pre(mx::T_W2);
  if ((st = mx_quantize(a->w2, 1, D, H, H, fmt, both, &w2_row, &w2t_row, nullptr, nullptr, 0, stream)) != MX_OK) return st;
  hk.post(mx::T_W2);
  hk.pre(mx::T_B1);
  if ((st = mx_gemm_gelu_fwd(&x_row, &w1_row, a->b1, pre, &act_row, &act_col, stream)) != MX_OK) return st;
  hk.post(mx::T_B1);
  hk.pre(mx::T_B2);
  hk.pre(mx::T_Y);
  if ((st = D % 256 == 0 ? pair_gemm_impl(&act_row, &w2_row, 1, nullptr, a->b2, 0, a->y, D, stream)
                          : mx_gemm_bias(&act_row, &w2_row, a->b2, a->y, D, stream)) != MX_OK)
    return st;
  hk.post(mx::T_B2);
  hk.post(mx::T_Y);
  hk.pre(mx::T_DY);
  hk.pre(mx::T_DB2);
  if ((st = mx_quantize(a->dy, 1, M, D, D, fmt, both | MX_COLSUM, &dy_row, &dy_col, a->db2, base + L.part_dy,
                        part_dy_bytes, stream)) != MX_OK)
    return st;
  hk.post(mx::T_DY);
  hk.post(mx::T_DB2);
  hk.pre(mx::T_DB1);
  if ((st = mx_gemm_dgelu_bwd(&dy_row, &w2t_row, pre, &dpre_row, &dpre_col, a->db1, base + L.part_dz,
                              part_dz_bytes, stream)) != MX_OK)
    return st;
  hk.post(mx::T_DB1);
  hk.pre(mx::T_DX);
  if ((st = plain_gemm(&dpre_row, &w1t_row, 1, nullptr, a->dx, D, stream)) != MX_OK) return st;
  hk.post(mx::T_DX);
  hk.pre(mx::T_DW2);
  // dense weight gradients: the same K order as the wgrad kernel's, as plain
  // GEMMs on CTA pairs where the widths allow (dW2 [D, H] = dY^T act, dW1
  // [H, D] = dpre^T X over the M tokens)
  if ((st = H % 256 == 0 ? plain_gemm(&dy_col, &act_col, 1, nullptr, a->dw2, H, stream)
                         : mx_grouped_gemm_wgrad(&dy_col, &act_col, 1, nullptr, a->dw2, stream)) != MX_OK)
    return st;
  hk.post(mx::T_DW2);
  hk.pre(mx::T_DW1);
  if ((st = D % 256 == 0 ? plain_gemm(&dpre_col, &x_col, 1, nullptr, a->dw1, D, stream)
                         : mx_grouped_gemm_wgrad(&dpre_col, &x_col, 1, nullptr, a->dw1, stream)) != MX_OK)
    return st;
  hk.post(mx::T_DW1);
  return MX_OK;
}

}  // namespace

size_t mx_mlp_workspace_bytes(const mx_mlp_args_t* args) {
  if (!args || args->R < 0 || args->D <= 0 || args->F <= 0 || args->G <= 0) return 0;
  if (args->fmt < MX_E4M3 || args->fmt > MX_E2M1) return 0;
  return mlp_layout(args).total;
}

mx_status_t mx_mlp_workspace_layout(const mx_mlp_args_t* args, mx_mlp_layout_t* out) {
  MX_CHECK(out != nullptr, MX_ERR_INVALID_ARG, "out is NULL");
  MX_CHECK(mx_mlp_workspace_bytes(args) > 0, MX_ERR_INVALID_ARG, "args is NULL or describes no valid step");
  const MlpLayout L = mlp_layout(args);
  auto put = [](const MlpLayout::Slot& s) {
    mx_mlp_slot_t o;
    o.data = s.data; o.scale = s.scale; o.rows = s.rows; o.cols = s.cols;
    return o;
  };
  out->x_row = put(L.x_row); out->x_col = put(L.x_col);
  out->w1_row = put(L.w1_row); out->w1t_row = put(L.w1t_row);
  out->w2_row = put(L.w2_row); out->w2t_row = put(L.w2t_row);
  out->h_row = put(L.h_row); out->h_col = put(L.h_col);
  out->dy_row = put(L.dy_row); out->dy_col = put(L.dy_col);
  out->dz_row = put(L.dz_row); out->dz_col = put(L.dz_col);
  out->z = L.z;
  out->total = L.total;
  return MX_OK;
}

}  // extern "C"

namespace mx {

// Validation shared by mx_mlp_fwd_bwd and the host pipeline.
mx_status_t mlp_check(const mx_mlp_args_t* a) {
  MX_CHECK(a != nullptr, MX_ERR_INVALID_ARG, "args is NULL");
  MX_CHECK(a->act == MX_ACT_SWIGLU || a->act == MX_ACT_GELU_TANH, MX_ERR_INVALID_ARG, "activation %d", a->act);
  if (a->act == MX_ACT_SWIGLU) {
    MX_CHECK(a->fmt == MX_E4M3 && a->hadamard == 0, MX_ERR_NOT_SUPPORTED,
             "the SwiGLU expert step runs on unrotated E4M3 operands");
  } else {
    MX_CHECK(a->fmt == MX_E4M3 || a->fmt == MX_E2M3, MX_ERR_NOT_SUPPORTED, "the GELU step runs on E4M3 or E2M3");
    MX_CHECK(a->G == 1, MX_ERR_NOT_SUPPORTED, "the GELU step is dense (G == 1)");
    MX_CHECK(a->db1 != nullptr && a->db2 != nullptr, MX_ERR_INVALID_ARG, "db1 and db2 are required");
  }
  MX_CHECK(a->G >= 1, MX_ERR_INVALID_ARG, "G = %d; at least one expert is required", a->G);
  MX_CHECK(a->R >= 0 && a->R % 128 == 0, MX_ERR_SHAPE, "R = %lld is not a multiple of 128", (long long)a->R);
  MX_CHECK(a->D > 0 && a->D % 128 == 0, MX_ERR_SHAPE, "D = %lld is not a positive multiple of 128", (long long)a->D);
  MX_CHECK(a->F > 0 && a->F % 128 == 0, MX_ERR_SHAPE, "F = %lld is not a positive multiple of 128", (long long)a->F);
  const void* ptrs[] = {a->x, a->w1, a->w2, a->dy, a->y, a->dx, a->dw1, a->dw2, a->workspace};
  const char* names[] = {"x", "w1", "w2", "dy", "y", "dx", "dw1", "dw2", "workspace"};
  for (int i = 0; i < 9; i++) {
    MX_CHECK(ptrs[i] != nullptr, MX_ERR_INVALID_ARG, "%s is NULL", names[i]);
    MX_CHECK(aligned16(ptrs[i]), MX_ERR_ALIGNMENT, "%s must be 16-byte aligned", names[i]);
  }
  const MlpLayout L = mlp_layout(a);
  MX_CHECK(a->workspace_bytes >= L.total, MX_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", L.total,
           a->workspace_bytes);
  return MX_OK;
}

mx_status_t mlp_step(const mx_mlp_args_t* a, mx_stream_t stream, const StepHooks* hooks) {
  mx_status_t st;
  if ((st = mlp_check(a)) != MX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = check_offsets(a->offsets, a->G, a->R, s)) != MX_OK) return st;
  if (a->R == 0) return MX_OK;
  const MlpLayout L = mlp_layout(a);
  return a->act == MX_ACT_SWIGLU ? mlp_swiglu(a, L, stream, hooks) : mlp_gelu(a, L, stream, hooks);
}

}  // namespace mx

extern "C" {

mx_status_t mx_mlp_fwd_bwd(const mx_mlp_args_t* a, mx_stream_t stream) { return mx::mlp_step(a, stream, nullptr); }

mx_status_t mx_get_device_status(mx_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0, dense = 0, f4 = 0, quant = 0, perm = 0, pairs = 0;
  if ((e = mx::read_gemm_status(&word)) != cudaSuccess || (e = mx::read_dense_status(&dense)) != cudaSuccess ||
      (e = mx::read_f4_status(&f4)) != cudaSuccess || (e = mx::read_quant_status(&quant)) != cudaSuccess ||
      (e = mx::read_perm_status(&perm)) != cudaSuccess || (e = mx::read_pair_status(&pairs)) != cudaSuccess)
    return cuda_fail(e, "reading device status");
  if ((e = mx::reset_gemm_status()) != cudaSuccess || (e = mx::reset_dense_status()) != cudaSuccess ||
      (e = mx::reset_f4_status()) != cudaSuccess || (e = mx::reset_quant_status()) != cudaSuccess ||
      (e = mx::reset_perm_status()) != cudaSuccess || (e = mx::reset_pair_status()) != cudaSuccess)
    return cuda_fail(e, "clearing device status");
  word |= dense | f4 | quant | perm | pairs;
  if (word & 1u) return fail(MX_ERR_DEVICE_TIMEOUT, "a bounded device-side wait expired");
  if (word & 2u) return fail(MX_ERR_OFFSETS, "a kernel saw a malformed offsets segment");
  if (word & 4u) return fail(MX_ERR_INVALID_ARG, "a routing index (expert id or routed row) was out of range");
  return MX_OK;
}

mx_status_t mx_debug_tap(float* tap_f32, int64_t elems) {
  MX_CHECK(tap_f32 == nullptr || (aligned16(tap_f32) && elems >= 0), MX_ERR_ALIGNMENT,
           "debug tap must be a 16-byte aligned pointer");
  g_tap = tap_f32;
  g_tap_elems = tap_f32 ? elems : 0;
  return MX_OK;
}

mx_status_t mx_selftest_bounded_wait(uint64_t budget_ns, mx_stream_t stream) {
  DevInfo dev;
  mx_status_t st = device_info(&dev);
  if (st != MX_OK) return st;
  MX_CHECK(budget_ns > 0 && budget_ns <= 2000000000ull, MX_ERR_INVALID_ARG, "budget must be in (0, 2 s]");
  cudaError_t e = mx::launch_wait_selftest(budget_ns, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return MX_OK;
}

}  // extern "C"
