"""CPU oracle for the OCP-MX training MLP -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links or
calls it, and it never imports the product package.

What it computes, and from which passage (web pages cited by title):

* Element codecs, exact RCEIL E8M0 scales, the blocked scale layout, packing
  and the 32-point Hadamard rotation live in ``mx_oracle.c`` (plain C,
  float64), wrapped here.  See that file's header for the readings it fixes.
* GEMMs are float64 matrix products of the *dequantized* operands
  (torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
  group gemm", shared-infrastructure commit: ragged grouped GEMM where each
  128-row-aligned segment uses its expert's weights; ragged-K wgrad where an
  expert with zero tokens gets a zero gradient).
* SwiGLU: h = g * sigmoid(g) * u with z = [g | u] the concatenated FC1
  halves, sigmoid = 1/(1+exp(-x)) (same PR, correctness-first kernels
  commit); dSwiGLU is its derivative, taken from the BF16-saved z.
* tanh-GELU MLP with bias added to the fp32 accumulator before one rounding
  (Primus PR #1064 "feat(mxfp6): MXFP6 (E2M3) Flux linears, a fused MLP, and
  the MLPerf recipe", fused-MLP and bias-in-epilogue commits).

Where floating point decides a quantized code inside a fused epilogue, the
oracle rounds the float64 value to fp32 first -- the arithmetic type the
epilogue quantizes from -- and then quantizes exactly.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

E4M3, E2M3, E2M1 = 0, 1, 2
FMT_NAMES = {E4M3: "e4m3", E2M3: "e2m3", E2M1: "e2m1"}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64 = ctypes.c_int64
        L.orc_decode.restype = ctypes.c_double
        L.orc_decode.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.orc_encode.restype = ctypes.c_uint8
        L.orc_encode.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_fmt_max.restype = ctypes.c_double
        L.orc_fmt_max.argtypes = [ctypes.c_int]
        L.orc_fmt_bits.restype = ctypes.c_int
        L.orc_fmt_bits.argtypes = [ctypes.c_int]
        L.orc_scale_exp.restype = ctypes.c_int
        L.orc_scale_exp.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_scale_byte.restype = ctypes.c_uint8
        L.orc_scale_byte.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_amax.restype = ctypes.c_double
        L.orc_amax.argtypes = [dp, i64]
        L.orc_quantize_block.restype = ctypes.c_uint8
        L.orc_quantize_block.argtypes = [dp, ctypes.c_int, u8p]
        L.orc_scale_bytes.restype = i64
        L.orc_scale_bytes.argtypes = [i64, i64]
        L.orc_blocked_offset.restype = i64
        L.orc_blocked_offset.argtypes = [i64, i64, i64]
        L.orc_payload_row_bytes.restype = i64
        L.orc_payload_row_bytes.argtypes = [i64, ctypes.c_int]
        L.orc_pack_row.argtypes = [u8p, i64, ctypes.c_int, u8p]
        L.orc_unpack_row.argtypes = [u8p, i64, ctypes.c_int, u8p]
        L.orc_hadamard32_f32.argtypes = [fp]
        L.orc_hadamard32_f64.argtypes = [dp, dp]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_quantize_rows.argtypes = [dp, i64, i64, ctypes.c_int, ctypes.c_int, u8p, u8p]
        L.orc_dequantize_rows.argtypes = [u8p, u8p, i64, i64, ctypes.c_int, dp]
        L.orc_bf16_to_f64_array.argtypes = [u16p, i64, dp]
        L.orc_f64_to_bf16_array.argtypes = [dp, i64, u16p]
        L.orc_round_f32_array.argtypes = [dp, i64, dp]
        u32p = ctypes.POINTER(ctypes.c_uint32)
        L.orc_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.orc_sr_bits.restype = ctypes.c_uint32
        L.orc_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        L.orc_encode_sr.restype = ctypes.c_uint8
        L.orc_encode_sr.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_uint32]
        L.orc_quantize_rows_sr.argtypes = [dp, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                           ctypes.c_uint32, u8p, u8p]
        _lib = L
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# --------------------------------------------------------------------------
# Scalar codecs
# --------------------------------------------------------------------------

def encode(v, fmt):
    return int(lib().orc_encode(float(v), fmt))


def decode(code, fmt):
    return float(lib().orc_decode(int(code), fmt))


def fmt_max(fmt):
    return float(lib().orc_fmt_max(fmt))


def scale_exp(amax, fmt):
    return int(lib().orc_scale_exp(float(amax), fmt))


def scale_byte(amax, fmt):
    return int(lib().orc_scale_byte(float(amax), fmt))


def quantize_block(x, fmt):
    """One block of 32 float64 values -> (scale byte, 32 unpacked codes)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    assert x.shape == (32,)
    codes = np.zeros(32, dtype=np.uint8)
    sb = lib().orc_quantize_block(_ptr(x, ctypes.c_double), fmt, _ptr(codes, ctypes.c_uint8))
    return int(sb), codes


def blocked_offset(r, c, scale_cols):
    return int(lib().orc_blocked_offset(r, c, scale_cols))


def scale_bytes(rows, scale_cols):
    return int(lib().orc_scale_bytes(rows, scale_cols))


def payload_row_bytes(cols, fmt):
    return int(lib().orc_payload_row_bytes(cols, fmt))


def hadamard32_f32(v):
    v = np.array(v, dtype=np.float32).copy()
    lib().orc_hadamard32_f32(_ptr(v, ctypes.c_float))
    return v


def hadamard32_f64(v):
    x = np.ascontiguousarray(v, dtype=np.float64)
    y = np.zeros(32, dtype=np.float64)
    lib().orc_hadamard32_f64(_ptr(x, ctypes.c_double), _ptr(y, ctypes.c_double))
    return y


# --------------------------------------------------------------------------
# Array conversions
# --------------------------------------------------------------------------

def bf16_to_f64(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().orc_bf16_to_f64_array(_ptr(bits, ctypes.c_uint16), bits.size, _ptr(out, ctypes.c_double))
    return out


def f64_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_array(_ptr(x, ctypes.c_double), x.size, _ptr(out, ctypes.c_uint16))
    return out


def round_f32(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    lib().orc_round_f32_array(_ptr(x, ctypes.c_double), x.size, _ptr(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------
# Whole-tensor quantization
# --------------------------------------------------------------------------

def quantize_rows(x, fmt, hadamard=False):
    """Rowwise 1x32 quantization of float64 [rows, cols].

    Returns (payload uint8 [rows, payload_row_bytes], scales uint8 blocked)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, cols = x.shape
    assert cols % 32 == 0
    payload = np.zeros((rows, payload_row_bytes(cols, fmt)), dtype=np.uint8)
    scales = np.zeros(scale_bytes(rows, cols // 32), dtype=np.uint8)
    lib().orc_quantize_rows(_ptr(x, ctypes.c_double), rows, cols, fmt, 1 if hadamard else 0,
                            _ptr(payload, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return payload, scales


def quantize_cols(x, fmt, hadamard=False):
    """Columnwise 32x1 quantization of [rows, cols]: blocks of 32 rows, stored
    as the rowwise quantization of the transpose, payload [cols, rows]."""
    return quantize_rows(np.ascontiguousarray(np.asarray(x, dtype=np.float64).T), fmt, hadamard)


def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC 2011) of a 4-word counter and a
    2-word key; returns the 4 output words."""
    c = (ctypes.c_uint32 * 4)(*counter)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    lib().orc_philox4x32_10(c, k, o)
    return tuple(int(v) for v in o)


def sr_bits(seed, idx, orient):
    return int(lib().orc_sr_bits(int(seed), int(idx), int(orient)))


def encode_sr(v, fmt, u):
    return int(lib().orc_encode_sr(float(v), fmt, int(u)))


def quantize_rows_sr(x, fmt, seed, orient=0, hadamard=False):
    """quantize_rows with stochastic rounding of the elements (scales stay
    RCEIL); element (r, c) draws its bits at index r * cols + c of this
    matrix with the given orientation word."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, cols = x.shape
    assert cols % 32 == 0
    payload = np.zeros((rows, payload_row_bytes(cols, fmt)), dtype=np.uint8)
    scales = np.zeros(scale_bytes(rows, cols // 32), dtype=np.uint8)
    lib().orc_quantize_rows_sr(_ptr(x, ctypes.c_double), rows, cols, fmt, 1 if hadamard else 0, int(seed),
                               int(orient), _ptr(payload, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return payload, scales


def quantize_cols_sr(x, fmt, seed, hadamard=False):
    """Columnwise quantization with stochastic rounding: the transpose
    [cols, rows] quantized rowwise with orientation word 1."""
    return quantize_rows_sr(np.ascontiguousarray(np.asarray(x, dtype=np.float64).T), fmt, seed, 1, hadamard)


def dequantize_rows(payload, scales, rows, cols, fmt):
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_dequantize_rows(_ptr(payload, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                              rows, cols, fmt, _ptr(out, ctypes.c_double))
    return out


def blocked_index(rows, scale_cols, row_ids=None):
    """int64 [rows, scale_cols] array of blocked-layout byte offsets (or
    [len(row_ids), scale_cols] for the given rows only)."""
    r = (np.arange(rows, dtype=np.int64) if row_ids is None else np.asarray(row_ids, dtype=np.int64))[:, None]
    c = np.arange(scale_cols, dtype=np.int64)[None, :]
    cpad = (scale_cols + 3) // 4 * 4
    # same closed form as orc_blocked_offset, vectorised; tests check they agree
    return ((r // 128) * (cpad // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def scales_to_matrix(scales, rows, scale_cols):
    """Blocked scale bytes -> logical [rows, scale_cols] matrix."""
    return np.asarray(scales, dtype=np.uint8)[blocked_index(rows, scale_cols)]


def quantize_bf16(x_bits, fmt, row=True, col=True, hadamard=False):
    """Quantize a BF16 tensor [R, C] (or a batch [B, R, C]) in one or both
    orientations.  Column outputs are per batch entry: payload [B, C, R']."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    batched = x_bits.ndim == 3
    xb = x_bits if batched else x_bits[None]
    out = {"row_payload": [], "row_scales": [], "col_payload": [], "col_scales": []}
    for b in range(xb.shape[0]):
        x = bf16_to_f64(xb[b])
        if row:
            p, s = quantize_rows(x, fmt, hadamard)
            out["row_payload"].append(p)
            out["row_scales"].append(s)
        if col:
            p, s = quantize_cols(x, fmt, hadamard)
            out["col_payload"].append(p)
            out["col_scales"].append(s)
    res = {}
    for k, v in out.items():
        if v:
            res[k] = np.stack(v) if batched else v[0]
    return res


def colsum(x):
    """Per-column sum over rows of a float64 [rows, cols] array (bias gradient)."""
    return np.asarray(x, dtype=np.float64).sum(axis=0)


# --------------------------------------------------------------------------
# GEMMs on dequantized operands (float64)
# --------------------------------------------------------------------------

def segments(offsets):
    """Cumulative end offsets -> list of (start, end)."""
    out, start = [], 0
    for end in np.asarray(offsets, dtype=np.int64).tolist():
        out.append((start, int(end)))
        start = int(end)
    return out


def grouped_gemm(a, b, offsets):
    """out[r, n] = sum_k a[r, k] * b[g, n, k] for r in expert g's segment.

    a float64 [R, K]; b float64 [G, N, K]; rows past offsets[-1] are NaN
    (never produced)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    out = np.full((a.shape[0], b.shape[1]), np.nan)
    for g, (s, e) in enumerate(segments(offsets)):
        if e > s:
            out[s:e] = a[s:e] @ b[g].T
    return out


def grouped_gemm_bias(a, b, bias, offsets):
    """grouped_gemm plus expert g's bias row on the rows of its segment:
    out[r, n] = sum_k a[r, k] * b[g, n, k] + bias[g, n] (Primus PR #1064
    "feat(mxfp6): MXFP6 (E2M3) Flux linears, a fused MLP, and the MLPerf
    recipe", bias commits: the bias joins the fp32 accumulator before the
    output's single rounding).  bias float64 [G, N]."""
    out = grouped_gemm(a, b, offsets)
    bias = np.asarray(bias, dtype=np.float64)
    for g, (s, e) in enumerate(segments(offsets)):
        if e > s:
            out[s:e] += bias[g][None, :]
    return out


def wgrad(a_col, b_col, offsets):
    """dW[g, n, k] = sum over r in segment g of a_col[n, r] * b_col[k, r].

    a_col float64 [N, R], b_col float64 [K, R] (columnwise operands stored
    transposed).  An empty segment gives an exactly zero slice."""
    a_col = np.asarray(a_col, dtype=np.float64)
    b_col = np.asarray(b_col, dtype=np.float64)
    segs = segments(offsets)
    out = np.zeros((len(segs), a_col.shape[0], b_col.shape[0]))
    for g, (s, e) in enumerate(segs):
        if e > s:
            out[g] = a_col[:, s:e] @ b_col[:, s:e].T
    return out


# --------------------------------------------------------------------------
# Token permute and un-permute (Primus PR #1247 "Qwen3-30B-A3B FP8 on MI355X
# to 40k tokens/s/GPU", DeepEP permute section: the dispatched tokens are
# quantized as part of the permute that hands them to the grouped MLP, and
# the un-permute's backward hands back the quantized output gradient).
# Readings where the page is silent: routed rows are grouped by expert in
# ascending expert order, within an expert in (token, choice) order; every
# expert's segment is padded with empty rows to a multiple of 128 (the
# grouped GEMM's segment alignment); an empty row is all zeros.
# --------------------------------------------------------------------------

def moe_route_index(topk, G, pad=128):
    """topk int [T, k] expert ids -> (offsets [G] cumulative padded segment
    ends, src [R] token of each routed row or -1 for a padding row with
    R = offsets[-1], row_of [T, k] routed row of each (token, choice))."""
    topk = np.asarray(topk)
    T, k = topk.shape
    members = [[] for _ in range(G)]
    for t in range(T):
        for j in range(k):
            e = int(topk[t, j])
            if not 0 <= e < G:
                raise ValueError("expert id %d out of range" % e)
            members[e].append((t, j))
    offsets = np.zeros(G, dtype=np.int32)
    src = []
    row_of = np.full((T, k), -1, dtype=np.int32)
    for e in range(G):
        for t, j in members[e]:
            row_of[t, j] = len(src)
            src.append(t)
        while len(src) % pad:
            src.append(-1)
        offsets[e] = len(src)
    return offsets, np.array(src, dtype=np.int32), row_of


def permute_rows(x, src):
    """out[r] = x[src[r]], or a zero row where src[r] < 0 (any dtype; BF16
    bit patterns give +0.0 rows)."""
    x = np.asarray(x)
    src = np.asarray(src)
    out = np.zeros((len(src),) + x.shape[1:], dtype=x.dtype)
    for r, t in enumerate(src.tolist()):
        if t >= 0:
            out[r] = x[t]
    return out


def permute_quantize(x_bits, src, fmt=E4M3, row=True, col=True):
    """The quantized permute: the routed rows of BF16 x, quantized in the
    permuted order (rowwise blocks along D, columnwise blocks of 32 routed
    rows)."""
    return quantize_bf16(permute_rows(x_bits, src), fmt, row, col)


def unpermute(y, row_of, weights=None):
    """out[t] = sum over choices j with row_of[t, j] >= 0 of
    w[t, j] * y[row_of[t, j]] (w = 1 without weights), float64: the
    combine after the experts, and the backward of the permute."""
    y = np.asarray(y, dtype=np.float64)
    row_of = np.asarray(row_of)
    T, k = row_of.shape
    out = np.zeros((T,) + y.shape[1:])
    for t in range(T):
        for j in range(k):
            r = int(row_of[t, j])
            if r >= 0:
                out[t] += (1.0 if weights is None else float(weights[t, j])) * y[r]
    return out


# --------------------------------------------------------------------------
# Activations (float64)
# --------------------------------------------------------------------------

def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def swiglu(g, u):
    return g * sigmoid(g) * u


def dswiglu(dh, g, u):
    s = sigmoid(g)
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    return dg, du


_GELU_C = math.sqrt(2.0 / math.pi)


def gelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(_GELU_C * (x + 0.044715 * x ** 3)))


def dgelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    t = np.tanh(_GELU_C * (x + 0.044715 * x ** 3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * _GELU_C * (1.0 + 3 * 0.044715 * x * x)


# --------------------------------------------------------------------------
# Fused stages: what each library call computes
# --------------------------------------------------------------------------

def _active_rows(offsets):
    return int(np.asarray(offsets, dtype=np.int64)[-1]) if len(offsets) else 0


def swiglu_fwd(x_deq, w1_deq, offsets, fmt=E4M3, probs=None):
    """FC1 grouped GEMM + SwiGLU + dual requant + BF16 pre-activation save.

    x_deq float64 [R, D] (dequantized rowwise X), w1_deq float64 [G, 2F, D].
    probs (optional) float [R]: each routed row's routing probability,
    multiplied into its activation row (Primus PR #1247 "Qwen3-30B-A3B FP8 on
    MI355X to 40k tokens/s/GPU": the fused activation with probabilities).
    Returns z (float64), z_bf16 (uint16 bits), h (fp32-rounded float64),
    h_row (payload, scales) over the active rows, h_col (payload, scales) of
    [F, A] where A = offsets[-1]."""
    A = _active_rows(offsets)
    z = grouped_gemm(x_deq, w1_deq, offsets)
    F = z.shape[1] // 2
    za = z[:A]
    act = swiglu(za[:, :F], za[:, F:])
    if probs is not None:
        act = act * np.asarray(probs, dtype=np.float64)[:A, None]
    h = round_f32(act)
    return {
        "z": z,
        "z_bf16": f64_to_bf16(za),
        "h": h,
        "h_row": quantize_rows(h, fmt),
        "h_col": quantize_cols(h, fmt),
    }


def dswiglu_bwd(dy_deq, w2t_deq, z_bf16, offsets, fmt=E4M3, probs=None):
    """FC2 dgrad grouped GEMM + dSwiGLU from the BF16-saved z + dual requant.

    dy_deq float64 [R, D]; w2t_deq float64 [G, F, D]; z_bf16 uint16 [>=A, 2F].
    With probs [R] (the forward scaled row r of the activation by p_r): the
    activation gradient is dh * p_r, and dprobs_r = sum_f dh[r, f] *
    swiglu(g, u)[r, f].
    Returns dh (float64), dz = [dg | du] (fp32-rounded), dz_row, dz_col, and
    dprobs (float64 [A]) when probs is given."""
    A = _active_rows(offsets)
    dh = grouped_gemm(dy_deq, w2t_deq, offsets)[:A]
    z = bf16_to_f64(np.asarray(z_bf16)[:A])
    F = dh.shape[1]
    g, u = z[:, :F], z[:, F:]
    out = {"dh": dh}
    if probs is not None:
        p = np.asarray(probs, dtype=np.float64)[:A, None]
        out["dprobs"] = np.sum(dh * swiglu(g, u), axis=1)
        dh = dh * p
    dg, du = dswiglu(dh, g, u)
    dz = round_f32(np.concatenate([dg, du], axis=1))
    out.update({"dz": dz, "dz_row": quantize_rows(dz, fmt), "dz_col": quantize_cols(dz, fmt)})
    return out


def bf16_out(x):
    """float64 -> BF16 bits -> float64 (the value a BF16 output holds)."""
    return bf16_to_f64(f64_to_bf16(x))


def quantize_experts_cols(w_bits, fmt=E4M3):
    """Per-expert columnwise quantization of BF16 weights [G, N, K]: each
    expert's transpose [K, N] rowwise; returns (payload [G*K, N'], scales of
    the stacked [G*K, N/32] matrix, blocked per expert)."""
    w_bits = np.asarray(w_bits, dtype=np.uint16)
    ps, ss = [], []
    for g in range(w_bits.shape[0]):
        p, s = quantize_cols(bf16_to_f64(w_bits[g]), fmt)
        ps.append(p)
        ss.append(s)
    return np.concatenate(ps), np.concatenate(ss)


def quantize_experts_rows(w_bits, fmt=E4M3):
    w_bits = np.asarray(w_bits, dtype=np.uint16)
    G, N, K = w_bits.shape
    return quantize_rows(bf16_to_f64(w_bits.reshape(G * N, K)), fmt)


def mlp_fwd_bwd_swiglu(x_bits, w1_bits, w2_bits, dy_bits, offsets, fmt=E4M3):
    """The whole MX SwiGLU expert-MLP step, stage by stage, each stage on the
    oracle's own quantization of its inputs.

    x [R, D], w1 [G, 2F, D], w2 [G, D, F], dy [R, D] as BF16 bits.  Returns a
    dict with every intermediate and the BF16-rounded outputs y, dx [R, D],
    dw1 [G, 2F, D], dw2 [G, D, F] (float64 values of the BF16 results)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    G, F2, D = np.asarray(w1_bits).shape
    F = F2 // 2
    R = x_bits.shape[0]
    A = _active_rows(offsets)
    x = bf16_to_f64(x_bits)
    dy = bf16_to_f64(dy_bits)
    x_row = quantize_rows(x, fmt)
    x_col = quantize_cols(x[:A], fmt)
    w1_row = quantize_experts_rows(w1_bits, fmt)
    w1t_row = quantize_experts_cols(w1_bits, fmt)
    w2_row = quantize_experts_rows(w2_bits, fmt)
    w2t_row = quantize_experts_cols(w2_bits, fmt)
    dq = lambda t, rows, cols: dequantize_rows(t[0], t[1], rows, cols, fmt)
    xq = dq(x_row, R, D)
    w1q = dq(w1_row, G * 2 * F, D).reshape(G, 2 * F, D)
    w1tq = dq(w1t_row, G * D, 2 * F).reshape(G, D, 2 * F)
    w2q = dq(w2_row, G * D, F).reshape(G, D, F)
    w2tq = dq(w2t_row, G * F, D).reshape(G, F, D)
    fwd = swiglu_fwd(xq, w1q, offsets, fmt)
    hq = dq(fwd["h_row"], A, F)
    y = grouped_gemm(np.concatenate([hq, np.zeros((R - A, F))]), w2q, offsets)
    dy_row = quantize_rows(dy, fmt)
    dy_col = quantize_cols(dy[:A], fmt)
    dyq = dq(dy_row, R, D)
    bwd = dswiglu_bwd(dyq, w2tq, fwd["z_bf16"], offsets, fmt)
    dzq = dq(bwd["dz_row"], A, 2 * F)
    dx = grouped_gemm(np.concatenate([dzq, np.zeros((R - A, 2 * F))]), w1tq, offsets)
    dyc = dq(dy_col, D, A)
    hc = dq(fwd["h_col"], F, A)
    dzc = dq(bwd["dz_col"], 2 * F, A)
    xc = dq(x_col, D, A)
    dw2 = wgrad(dyc, hc, offsets)
    dw1 = wgrad(dzc, xc, offsets)
    return {
        "x_row": x_row, "x_col": x_col, "w1_row": w1_row, "w1t_row": w1t_row, "w2_row": w2_row,
        "w2t_row": w2t_row, "dy_row": dy_row, "dy_col": dy_col, "fwd": fwd, "bwd": bwd,
        "y": bf16_out(y[:A]), "dx": bf16_out(dx[:A]), "dw1": bf16_out(dw1), "dw2": bf16_out(dw2),
        "y_f64": y[:A], "dx_f64": dx[:A], "dw1_f64": dw1, "dw2_f64": dw2,
    }


def mlp_fwd_bwd_swiglu_unquantized(x_bits, w1_bits, w2_bits, dy_bits, offsets):
    """The same step in float64 with no quantization at all (the reference
    the quantized chain's SQNR is measured against), on BF16 inputs."""
    return mlp_fwd_bwd_swiglu_f64(bf16_to_f64(x_bits), bf16_to_f64(w1_bits), bf16_to_f64(w2_bits),
                                  bf16_to_f64(dy_bits), offsets)


def mlp_fwd_bwd_swiglu_f64(x, w1, w2, dy, offsets):
    """The unquantized SwiGLU expert-MLP step on float64 arrays: x [R, D],
    w1 [G, 2F, D], w2 [G, D, F], dy [R, D].  Rows past offsets[-1] take no
    part.  Forward z = x W1[g]^T, h = swiglu(z), y = h W2[g]^T; backward
    of the loss sum(y * dy): dh = dy W2[g], dz = dswiglu(dh, z),
    dx = dz W1[g], dW2[g] = dy_seg^T h_seg, dW1[g] = dz_seg^T x_seg."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    A = _active_rows(offsets)
    F = w1.shape[1] // 2
    z = grouped_gemm(x, w1, offsets)[:A]
    g, u = z[:, :F], z[:, F:]
    h = swiglu(g, u)
    R = x.shape[0]
    hp = np.concatenate([h, np.zeros((R - A, F))])
    y = grouped_gemm(hp, w2, offsets)[:A]
    dh = grouped_gemm(dy, np.transpose(w2, (0, 2, 1)), offsets)[:A]
    dg, du = dswiglu(dh, g, u)
    dz = np.concatenate([dg, du], axis=1)
    dzp = np.concatenate([dz, np.zeros((R - A, 2 * F))])
    dx = grouped_gemm(dzp, np.transpose(w1, (0, 2, 1)), offsets)[:A]
    dw2 = wgrad(dy[:A].T, h.T, offsets)
    dw1 = wgrad(dz.T, x[:A].T, offsets)
    return {"z": z, "h": h, "y": y, "dx": dx, "dw1": dw1, "dw2": dw2}


def sqnr_db(ref, test):
    ref = np.asarray(ref, dtype=np.float64)
    err = np.asarray(test, dtype=np.float64) - ref
    return 10.0 * np.log10(np.sum(ref * ref) / max(np.sum(err * err), 1e-300))


def within_tolerance(test, ref):
    """|test - ref| <= 2^-8 |ref| + 2^-14 rms(row of ref), elementwise."""
    ref = np.asarray(ref, dtype=np.float64)
    test = np.asarray(test, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * rms
    return np.abs(test - ref) <= bound


# --------------------------------------------------------------------------
# Dense MXFP6 + Hadamard + tanh-GELU MLP (Primus PR #1064)
# --------------------------------------------------------------------------

def gelu_fwd(x_deq, w1_deq, b1, fmt=E2M3, hadamard=True):
    """FC1 with bias in the accumulator, BF16 pre-activation save, and the
    tanh-GELU activation packed rowwise [M, H] and columnwise [H, M]."""
    pre = np.asarray(x_deq) @ np.asarray(w1_deq).T
    if b1 is not None:
        pre = pre + np.asarray(b1, dtype=np.float64)[None, :]
    act = round_f32(gelu_tanh(round_f32(pre)))
    return {"pre": pre, "pre_bf16": f64_to_bf16(pre), "act": act,
            "act_row": quantize_rows(act, fmt, hadamard), "act_col": quantize_cols(act, fmt, hadamard)}


def dgelu_bwd(dy_deq, w2t_deq, pre_bf16, fmt=E2M3, hadamard=True):
    """FC2 dgrad with the dGELU epilogue: dpre = (dY W2) * gelu'(pre) from
    the BF16-saved pre-activation, packed both ways, plus its column sums."""
    da = np.asarray(dy_deq) @ np.asarray(w2t_deq).T
    dpre64 = da * dgelu_tanh(bf16_to_f64(pre_bf16))
    dpre = round_f32(dpre64)
    return {"da": da, "dpre": dpre, "db1": colsum(dpre64),
            "dpre_row": quantize_rows(dpre, fmt, hadamard), "dpre_col": quantize_cols(dpre, fmt, hadamard)}


def mlp_fwd_bwd_gelu(x_bits, w1_bits, w2_bits, b1_bits, b2_bits, dy_bits, fmt=E2M3, hadamard=True):
    """The dense MX GELU MLP step, stage by stage on the oracle's own
    quantization: x [M, D], w1 [H, D], w2 [D, H], b1 [H], b2 [D], dy [M, D]."""
    x, dy = bf16_to_f64(x_bits), bf16_to_f64(dy_bits)
    w1, w2 = bf16_to_f64(w1_bits), bf16_to_f64(w2_bits)
    b1, b2 = bf16_to_f64(b1_bits), bf16_to_f64(b2_bits)
    M, D = x.shape
    H = w1.shape[0]
    dq = lambda t, rows, cols: dequantize_rows(t[0], t[1], rows, cols, fmt)
    x_row, x_col = quantize_rows(x, fmt, hadamard), quantize_cols(x, fmt, hadamard)
    w1_row, w1t_row = quantize_rows(w1, fmt, hadamard), quantize_cols(w1, fmt, hadamard)
    w2_row, w2t_row = quantize_rows(w2, fmt, hadamard), quantize_cols(w2, fmt, hadamard)
    fwd = gelu_fwd(dq(x_row, M, D), dq(w1_row, H, D), b1, fmt, hadamard)
    y = dq(fwd["act_row"], M, H) @ dq(w2_row, D, H).T + b2[None, :]
    dy_row, dy_col = quantize_rows(dy, fmt, hadamard), quantize_cols(dy, fmt, hadamard)
    db2 = colsum(dy)
    bwd = dgelu_bwd(dq(dy_row, M, D), dq(w2t_row, H, D), fwd["pre_bf16"], fmt, hadamard)
    dx = dq(bwd["dpre_row"], M, H) @ dq(w1t_row, D, H).T
    dw2 = dq(dy_col, D, M) @ dq(fwd["act_col"], H, M).T
    dw1 = dq(bwd["dpre_col"], H, M) @ dq(x_col, D, M).T
    return {"x_row": x_row, "x_col": x_col, "w1_row": w1_row, "w1t_row": w1t_row, "w2_row": w2_row,
            "w2t_row": w2t_row, "dy_row": dy_row, "dy_col": dy_col, "fwd": fwd, "bwd": bwd,
            "y_f64": y, "dx_f64": dx, "dw1_f64": dw1, "dw2_f64": dw2, "db1": bwd["db1"], "db2": db2}


def mlp_fwd_bwd_gelu_unquantized(x_bits, w1_bits, w2_bits, b1_bits, b2_bits, dy_bits):
    """The dense GELU MLP step in float64 with no quantization and no
    rotation, on BF16 inputs."""
    return mlp_fwd_bwd_gelu_f64(bf16_to_f64(x_bits), bf16_to_f64(w1_bits), bf16_to_f64(w2_bits),
                                bf16_to_f64(b1_bits), bf16_to_f64(b2_bits), bf16_to_f64(dy_bits))


def mlp_fwd_bwd_gelu_f64(x, w1, w2, b1, b2, dy):
    """The unquantized dense GELU MLP step on float64 arrays: x [M, D],
    w1 [H, D], w2 [D, H], b1 [H], b2 [D], dy [M, D].  Forward
    pre = x W1^T + b1, act = gelu_tanh(pre), y = act W2^T + b2; backward of
    the loss sum(y * dy): dpre = (dy W2) * gelu'(pre), dx = dpre W1,
    dW2 = dy^T act, dW1 = dpre^T x, db1 / db2 = column sums of dpre / dy."""
    x, dy = np.asarray(x, dtype=np.float64), np.asarray(dy, dtype=np.float64)
    w1, w2 = np.asarray(w1, dtype=np.float64), np.asarray(w2, dtype=np.float64)
    b1, b2 = np.asarray(b1, dtype=np.float64), np.asarray(b2, dtype=np.float64)
    pre = x @ w1.T + b1[None, :]
    act = gelu_tanh(pre)
    y = act @ w2.T + b2[None, :]
    dpre = (dy @ w2) * dgelu_tanh(pre)
    return {"pre": pre, "y": y, "dx": dpre @ w1, "dw2": dy.T @ act, "dw1": dpre.T @ x,
            "db1": dpre.sum(0), "db2": dy.sum(0)}
