/*
 * mx_oracle.c -- plain, slow, scalar CPU reference for the OCP-MX training MLP.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or table generator with the
 * CUDA library; every table here is derived from the format definitions below.
 *
 * Sources (web pages, cited by title and the passage within them):
 *   [MXFP4-guide]  ROCm Primus guide "MXFP4 training for Flux models",
 *                  Overview: block of 32 elements sharing one E8M0 exponent.
 *   [MXFP6-PR]     Primus PR #1064 "feat(mxfp6): MXFP6 (E2M3) Flux linears,
 *                  a fused MLP, and the MLPerf recipe", first commit message
 *                  (E2M3, mandatory Hadamard rotation folded into the packer)
 *                  and the bias commits (bias added in the fp32 accumulator).
 *   [MXFP8-PR]     torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP
 *                  fwd/bwd and wgrad group gemm": shared-infrastructure commit
 *                  (RCEIL E8M0, NaN-propagating amax, blocked-scale indexing,
 *                  512-byte K stride, whole-matrix columnwise scales) and the
 *                  correctness-first kernels commit (RCEIL, f32->E4M3 equal to
 *                  torch's cast, sigmoid as 1/(1+exp(-x))).
 *
 * Conventions fixed here where the pages are silent (each is a reading):
 *   - element formats follow the OCP MX element definitions: E4M3 (bias 7,
 *     max 448, NaN = S.1111.111, no Inf), E2M3 (bias 1, max 7.5, no NaN/Inf),
 *     E2M1 (bias 1, max 6.0, no NaN/Inf); E8M0 byte b means 2^(b-127), 0xFF NaN.
 *   - block scale: the smallest integer e with amax <= emax * 2^e ("RCEIL",
 *     i.e. the exact ceiling of log2(amax/emax)), clamped to [-127, 127].
 *     amax == 0 -> byte 0x00; amax == +Inf -> 0xFE; amax NaN -> 0xFF.
 *   - element encode: x * 2^-e rounded to nearest, ties to even code,
 *     saturating at +-emax; sign of zero kept.  A NaN block stores the
 *     format's NaN code (E4M3 0x7F) or +0 (E2M3, E2M1) in every element.
 *   - 32-point Hadamard: Sylvester order, orthonormal (H/sqrt(32)), evaluated
 *     in fp32 as five in-place butterfly stages (stride 1,2,4,8,16) followed by
 *     one multiply by fl32(1/sqrt(32)).  Parity unpinned beyond its algebra.
 *
 * Compile with -ffp-contract=off: the fp32 Hadamard sequence must not fuse.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

enum { ORC_E4M3 = 0, ORC_E2M3 = 1, ORC_E2M1 = 2 };

/* ----------------------------------------------------------------------- */
/* Element formats (OCP MX definitions, named by the pages).               */
/* ----------------------------------------------------------------------- */

typedef struct { int ebits, mbits, bias; int has_nan; } orc_fmt_desc;

static orc_fmt_desc fmt_desc(int fmt) {
  orc_fmt_desc d;
  if (fmt == ORC_E4M3) { d.ebits = 4; d.mbits = 3; d.bias = 7; d.has_nan = 1; }
  else if (fmt == ORC_E2M3) { d.ebits = 2; d.mbits = 3; d.bias = 1; d.has_nan = 0; }
  else { d.ebits = 2; d.mbits = 1; d.bias = 1; d.has_nan = 0; }
  return d;
}

int orc_fmt_bits(int fmt) { orc_fmt_desc d = fmt_desc(fmt); return 1 + d.ebits + d.mbits; }

/* Value of a code, from the sign / exponent / mantissa fields. */
double orc_decode(uint8_t code, int fmt) {
  orc_fmt_desc d = fmt_desc(fmt);
  int nbits = 1 + d.ebits + d.mbits;
  int sign = (code >> (nbits - 1)) & 1;
  int efield = (code >> d.mbits) & ((1 << d.ebits) - 1);
  int mfield = code & ((1 << d.mbits) - 1);
  if (d.has_nan && efield == (1 << d.ebits) - 1 && mfield == (1 << d.mbits) - 1) return NAN;
  double mag;
  if (efield == 0) mag = ldexp((double)mfield, 1 - d.bias - d.mbits);              /* subnormal */
  else mag = ldexp((double)((1 << d.mbits) + mfield), efield - d.bias - d.mbits);  /* normal */
  return sign ? -mag : mag;
}

/* Largest positive finite code (codes of one sign are ordered by value). */
static int max_pos_code(int fmt) {
  orc_fmt_desc d = fmt_desc(fmt);
  int top = (1 << (d.ebits + d.mbits)) - 1;  /* all exponent and mantissa bits set */
  return d.has_nan ? top - 1 : top;
}

double orc_fmt_max(int fmt) { return orc_decode((uint8_t)max_pos_code(fmt), fmt); }

/* Decoded values of the positive codes, filled once from orc_decode. */
static double g_tab[3][128];
static int g_tab_ready = 0;

void orc_init(void) {
  if (g_tab_ready) return;
  for (int f = 0; f < 3; f++)
    for (int c = 0; c <= max_pos_code(f); c++) g_tab[f][c] = orc_decode((uint8_t)c, f);
  g_tab_ready = 1;
}

/* Round-to-nearest, ties to the even code, saturating at +-max, sign of zero
 * kept.  Binary search over the ordered positive codes (0 .. max_pos_code). */
uint8_t orc_encode(double v, int fmt) {
  orc_init();
  orc_fmt_desc d = fmt_desc(fmt);
  int nbits = 1 + d.ebits + d.mbits;
  uint8_t sign_bit = (uint8_t)(1u << (nbits - 1));
  if (isnan(v)) return d.has_nan ? (uint8_t)((1 << (nbits - 1)) - 1) : 0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  const double *tab = g_tab[fmt];
  int hi = max_pos_code(fmt);
  int k;
  if (a >= tab[hi]) {
    k = hi;                                   /* saturate (includes +-Inf) */
  } else {
    int lo = 0, up = hi;                      /* tab[lo] <= a < tab[up] */
    while (up - lo > 1) {
      int mid = (lo + up) / 2;
      if (tab[mid] <= a) lo = mid; else up = mid;
    }
    double vlo = tab[lo], vup = tab[up];
    double midpoint = 0.5 * (vlo + vup);      /* exact in double */
    if (a < midpoint) k = lo;
    else if (a > midpoint) k = up;
    else k = (lo & 1) ? up : lo;              /* tie: the code whose LSB is 0 */
  }
  return (uint8_t)(k | (neg ? sign_bit : 0));
}

/* ----------------------------------------------------------------------- */
/* E8M0 block scale, round up (RCEIL).                                     */
/* ----------------------------------------------------------------------- */

/* Smallest integer e with a <= emax * 2^e, for finite a > 0 (unclamped). */
int orc_scale_exp(double a, int fmt) {
  double emax = orc_fmt_max(fmt);
  int e = ilogb(a) - ilogb(emax);
  while (a > ldexp(emax, e)) e++;
  while (a <= ldexp(emax, e - 1)) e--;
  return e;
}

/* Scale byte for a block whose NaN-propagating amax is `a`. */
uint8_t orc_scale_byte(double a, int fmt) {
  if (isnan(a)) return 0xFF;
  if (isinf(a)) return 0xFE;
  if (a == 0.0) return 0x00;
  int e = orc_scale_exp(a, fmt);
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return (uint8_t)(e + 127);
}

/* NaN-propagating max of |x| over n values. */
double orc_amax(const double *x, int64_t n) {
  double m = 0.0;
  for (int64_t i = 0; i < n; i++) {
    if (isnan(x[i])) return NAN;
    double a = fabs(x[i]);
    if (a > m) m = a;
  }
  return m;
}

/* Quantize one block of 32 values (already rotated if Hadamard is on):
 * writes 32 unpacked codes and returns the scale byte. */
uint8_t orc_quantize_block(const double *x, int fmt, uint8_t *codes) {
  double a = orc_amax(x, 32);
  uint8_t sb = orc_scale_byte(a, fmt);
  if (sb == 0xFF) {
    for (int i = 0; i < 32; i++) codes[i] = orc_encode(NAN, fmt);
    return sb;
  }
  int e = (int)sb - 127;
  for (int i = 0; i < 32; i++) codes[i] = orc_encode(ldexp(x[i], -e), fmt);
  return sb;
}

/* ----------------------------------------------------------------------- */
/* Stochastic rounding of the element step (Primus guide "MXFP4 training    */
/* for Flux models": optional stochastic rounding of the FP4 gradient        */
/* quantization).  The pages name the option only; our reading: the scale   */
/* stays RCEIL, and each scaled element rounds to one of its two grid        */
/* neighbours, up with probability equal to its fractional position.       */
/* Random bits: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random */
/* numbers: as easy as 1, 2, 3", SC 2011), counter-based, keyed by the seed. */
/* ----------------------------------------------------------------------- */

/* Ten rounds of the Philox 4x32 bijection: two 32x32->64 multiplies per
 * round, the key bumped by the Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; round++) {
    if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32 random bits of element `idx` of an output grid: counter
 * (idx / 4 as two words, orientation, 0), key = the seed's two words, word
 * idx % 4 of the result. */
uint32_t orc_sr_bits(uint64_t seed, uint64_t idx, uint32_t orient) {
  uint64_t n = idx >> 2;
  uint32_t ctr[4] = {(uint32_t)n, (uint32_t)(n >> 32), orient, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[idx & 3];
}

/* Stochastic encode of a scaled value v (an fp32 value): saturating at
 * +-max, otherwise the upper neighbour when (u >> 8) < frac * 2^24 with
 * frac = (|v| - lo) / (up - lo), which is exact (the spacing is a power of
 * two and |v| - lo is exact); the lower neighbour else.  Sign of zero kept;
 * NaN as orc_encode. */
uint8_t orc_encode_sr(double v, int fmt, uint32_t u) {
  orc_init();
  orc_fmt_desc d = fmt_desc(fmt);
  int nbits = 1 + d.ebits + d.mbits;
  uint8_t sign_bit = (uint8_t)(1u << (nbits - 1));
  if (isnan(v)) return d.has_nan ? (uint8_t)((1 << (nbits - 1)) - 1) : 0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  const double *tab = g_tab[fmt];
  int hi = max_pos_code(fmt);
  int k;
  if (a >= tab[hi]) {
    k = hi;
  } else {
    int lo = 0, up = hi;
    while (up - lo > 1) {
      int mid = (lo + up) / 2;
      if (tab[mid] <= a) lo = mid; else up = mid;
    }
    double frac = (a - tab[lo]) / (tab[up] - tab[lo]);
    k = ((double)(u >> 8) < frac * 16777216.0) ? up : lo;
  }
  return (uint8_t)(k | (neg ? sign_bit : 0));
}

/* One block with stochastic rounding: element i of the block is element
 * idx0 + i of the output grid.  The scaled value is rounded to fp32 first,
 * as the device's fp32 multiply does. */
uint8_t orc_quantize_block_sr(const double *x, int fmt, uint64_t seed, uint64_t idx0, uint32_t orient,
                              uint8_t *codes) {
  double a = orc_amax(x, 32);
  uint8_t sb = orc_scale_byte(a, fmt);
  if (sb == 0xFF) {
    for (int i = 0; i < 32; i++) codes[i] = orc_encode(NAN, fmt);
    return sb;
  }
  int e = (int)sb - 127;
  for (int i = 0; i < 32; i++) {
    double v = (double)(float)ldexp(x[i], -e);
    codes[i] = orc_encode_sr(v, fmt, orc_sr_bits(seed, idx0 + (uint64_t)i, orient));
  }
  return sb;
}

/* ----------------------------------------------------------------------- */
/* Blocked ("128x4") scale layout of the tcgen05 block-scaled MMA.          */
/* [MXFP8-PR] shared-infrastructure commit: tcgen05 blocked-scale indexing, */
/* constant 512-byte K stride for every 128-row block.                      */
/* ----------------------------------------------------------------------- */

static int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

/* Bytes of a blocked scale matrix for `rows` rows and `scale_cols` scales per row. */
int64_t orc_scale_bytes(int64_t rows, int64_t scale_cols) {
  return round_up(rows, 128) * round_up(scale_cols, 4);
}

int64_t orc_blocked_offset(int64_t r, int64_t c, int64_t scale_cols) {
  int64_t cpad = round_up(scale_cols, 4);
  return ((r / 128) * (cpad / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* ----------------------------------------------------------------------- */
/* Packing of codes into payload bytes.                                    */
/* E4M3: one byte each.  E2M1: two per byte, even index in the low nibble.  */
/* E2M3: four per three bytes, element i at bits [6i, 6i+6) of the          */
/* little-endian bit stream of each 3-byte group.                          */
/* ----------------------------------------------------------------------- */

int64_t orc_payload_row_bytes(int64_t cols, int fmt) {
  if (fmt == ORC_E4M3) return cols;
  if (fmt == ORC_E2M1) return cols / 2;
  return cols / 4 * 3;
}

void orc_pack_row(const uint8_t *codes, int64_t cols, int fmt, uint8_t *out) {
  if (fmt == ORC_E4M3) { memcpy(out, codes, (size_t)cols); return; }
  if (fmt == ORC_E2M1) {
    for (int64_t i = 0; i < cols / 2; i++)
      out[i] = (uint8_t)((codes[2 * i] & 0xF) | ((codes[2 * i + 1] & 0xF) << 4));
    return;
  }
  for (int64_t g = 0; g < cols / 4; g++) {
    uint32_t bits = 0;
    for (int j = 0; j < 4; j++) bits |= (uint32_t)(codes[4 * g + j] & 0x3F) << (6 * j);
    out[3 * g + 0] = (uint8_t)(bits & 0xFF);
    out[3 * g + 1] = (uint8_t)((bits >> 8) & 0xFF);
    out[3 * g + 2] = (uint8_t)((bits >> 16) & 0xFF);
  }
}

void orc_unpack_row(const uint8_t *in, int64_t cols, int fmt, uint8_t *codes) {
  if (fmt == ORC_E4M3) { memcpy(codes, in, (size_t)cols); return; }
  if (fmt == ORC_E2M1) {
    for (int64_t i = 0; i < cols / 2; i++) {
      codes[2 * i] = in[i] & 0xF;
      codes[2 * i + 1] = (in[i] >> 4) & 0xF;
    }
    return;
  }
  for (int64_t g = 0; g < cols / 4; g++) {
    uint32_t bits = (uint32_t)in[3 * g] | ((uint32_t)in[3 * g + 1] << 8) | ((uint32_t)in[3 * g + 2] << 16);
    for (int j = 0; j < 4; j++) codes[4 * g + j] = (uint8_t)((bits >> (6 * j)) & 0x3F);
  }
}

/* ----------------------------------------------------------------------- */
/* 32-point Hadamard rotation ([MXFP6-PR], first commit).                  */
/* ----------------------------------------------------------------------- */

/* fp32 evaluation in the fixed order the rotation is defined with here. */
void orc_hadamard32_f32(float *v) {
  for (int h = 1; h < 32; h <<= 1) {
    for (int i = 0; i < 32; i++) {
      if (i & h) continue;
      float a = v[i], b = v[i + h];
      v[i] = a + b;
      v[i + h] = a - b;
    }
  }
  const float inv = (float)(1.0 / sqrt(32.0));
  for (int i = 0; i < 32; i++) v[i] = v[i] * inv;
}

/* Exact definition in float64: y[i] = sum_j (-1)^popcount(i&j) x[j] / sqrt(32). */
void orc_hadamard32_f64(const double *x, double *y) {
  for (int i = 0; i < 32; i++) {
    double s = 0.0;
    for (int j = 0; j < 32; j++) {
      int p = __builtin_popcount((unsigned)(i & j)) & 1;
      s += p ? -x[j] : x[j];
    }
    y[i] = s / sqrt(32.0);
  }
}

/* ----------------------------------------------------------------------- */
/* BF16 <-> double.                                                        */
/* ----------------------------------------------------------------------- */

double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest BF16 (8-bit significand, fp32 exponent
 * range, subnormals down to 2^-133), ties to even; overflow to +-Inf. */
uint16_t orc_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  double r;
  if (isinf(a)) {
    r = INFINITY;
  } else if (a == 0.0) {
    r = 0.0;
  } else {
    int ex = ilogb(a);
    if (ex < -126) ex = -126;                 /* subnormal: fixed quantum */
    double q = ldexp(1.0, ex - 7);            /* spacing of BF16 values at a */
    r = nearbyint(a / q) * q;                 /* a/q is exact: q is a power of 2 */
    if (r >= ldexp(1.0, 128)) r = INFINITY;   /* rounds past the largest finite */
  }
  float f = (float)r;                         /* exact: r is a BF16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t b = (uint16_t)(u >> 16);
  return neg ? (uint16_t)(b | 0x8000) : b;
}

/* ----------------------------------------------------------------------- */
/* Whole-tensor quantization.                                              */
/* ----------------------------------------------------------------------- */

/* Rowwise 1x32: blocks of 32 consecutive columns of each row.  `x` is
 * double [rows, cols] (the values to quantize; BF16 inputs converted
 * exactly).  If `hadamard`, each block is first rotated with the fp32
 * sequence (input rounded to fp32 first).  Writes packed payload
 * [rows, payload_row_bytes] and blocked scales (zeroed padding). */
void orc_quantize_rows(const double *x, int64_t rows, int64_t cols, int fmt, int hadamard,
                       uint8_t *payload, uint8_t *scales) {
  int64_t sc = cols / 32;
  int64_t rb = orc_payload_row_bytes(cols, fmt);
  memset(scales, 0, (size_t)orc_scale_bytes(rows, sc));
  orc_init();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    uint8_t codes[32];
    uint8_t *rowcodes = (uint8_t *)__builtin_alloca((size_t)cols);
    for (int64_t b = 0; b < sc; b++) {
      double blk[32];
      if (hadamard) {
        float f[32];
        for (int i = 0; i < 32; i++) f[i] = (float)x[r * cols + b * 32 + i];
        orc_hadamard32_f32(f);
        for (int i = 0; i < 32; i++) blk[i] = (double)f[i];
      } else {
        for (int i = 0; i < 32; i++) blk[i] = x[r * cols + b * 32 + i];
      }
      scales[orc_blocked_offset(r, b, sc)] = orc_quantize_block(blk, fmt, codes);
      memcpy(rowcodes + b * 32, codes, 32);
    }
    orc_pack_row(rowcodes, cols, fmt, payload + r * rb);
  }
}

/* orc_quantize_rows with stochastic rounding; the element grid is this
 * [rows, cols] matrix (row-major index r * cols + c), `orient` the fourth
 * Philox counter word (0 for a rowwise output, 1 for a columnwise one). */
void orc_quantize_rows_sr(const double *x, int64_t rows, int64_t cols, int fmt, int hadamard, uint64_t seed,
                          uint32_t orient, uint8_t *payload, uint8_t *scales) {
  int64_t sc = cols / 32;
  int64_t rb = orc_payload_row_bytes(cols, fmt);
  memset(scales, 0, (size_t)orc_scale_bytes(rows, sc));
  orc_init();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    uint8_t codes[32];
    uint8_t *rowcodes = (uint8_t *)__builtin_alloca((size_t)cols);
    for (int64_t b = 0; b < sc; b++) {
      double blk[32];
      if (hadamard) {
        float f[32];
        for (int i = 0; i < 32; i++) f[i] = (float)x[r * cols + b * 32 + i];
        orc_hadamard32_f32(f);
        for (int i = 0; i < 32; i++) blk[i] = (double)f[i];
      } else {
        for (int i = 0; i < 32; i++) blk[i] = x[r * cols + b * 32 + i];
      }
      scales[orc_blocked_offset(r, b, sc)] =
          orc_quantize_block_sr(blk, fmt, seed, (uint64_t)(r * cols + b * 32), orient, codes);
      memcpy(rowcodes + b * 32, codes, 32);
    }
    orc_pack_row(rowcodes, cols, fmt, payload + r * rb);
  }
}

/* Dequantize a rowwise MX tensor back to double [rows, cols] (the rotation,
 * if any, is not undone: the GEMM consumes rotated operands). */
void orc_dequantize_rows(const uint8_t *payload, const uint8_t *scales, int64_t rows, int64_t cols,
                         int fmt, double *out) {
  int64_t sc = cols / 32;
  int64_t rb = orc_payload_row_bytes(cols, fmt);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    uint8_t *rowcodes = (uint8_t *)__builtin_alloca((size_t)cols);
    orc_unpack_row(payload + r * rb, cols, fmt, rowcodes);
    for (int64_t c = 0; c < cols; c++) {
      uint8_t sb = scales[orc_blocked_offset(r, c / 32, sc)];
      double v = orc_decode(rowcodes[c], fmt);
      out[r * cols + c] = (sb == 0xFF) ? NAN : ldexp(v, (int)sb - 127);
    }
  }
}

void orc_bf16_to_f64_array(const uint16_t *in, int64_t n, double *out) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_bf16_to_f64(in[i]);
}

void orc_f64_to_bf16_array(const double *in, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_f64_to_bf16(in[i]);
}

/* Round each double to the nearest fp32 (the epilogue's arithmetic type),
 * ties to even, as the C conversion does under the default rounding mode. */
void orc_round_f32_array(const double *in, int64_t n, double *out) {
  for (int64_t i = 0; i < n; i++) out[i] = (double)(float)in[i];
}
