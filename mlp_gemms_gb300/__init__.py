"""Thin Python binding of the GB300 MX training-MLP library (``include/mx.h``).

Argument marshalling only: every function here checks nothing the C layer
does not, computes nothing, and calls exactly one C-ABI entry point of the
same name (``mx_mlp_fwd_bwd`` launches the whole step).  PyTorch supplies
device memory (output buffers are ``torch.empty`` allocations when the
caller passes none) and the current CUDA stream.

There is no fallback: if the shared library is missing or fails to load,
``load()`` raises and nothing runs.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmxgb300.so")

E4M3, E2M3, E2M1 = 0, 1, 2
ROWWISE, COLWISE, HADAMARD, COLSUM = 1, 2, 4, 8
ACT_SWIGLU, ACT_GELU_TANH = 0, 1

STATUS = {
    0: "MX_OK", 1: "MX_ERR_INVALID_ARG", 2: "MX_ERR_SHAPE", 3: "MX_ERR_ALIGNMENT", 4: "MX_ERR_OFFSETS",
    5: "MX_ERR_UNSUPPORTED_DEVICE", 6: "MX_ERR_CUDA", 7: "MX_ERR_DEVICE_TIMEOUT", 8: "MX_ERR_WORKSPACE",
    9: "MX_ERR_NOT_SUPPORTED",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

# Every symbol include/mx.h declares.
ABI_SYMBOLS = (
    "mx_abi_version", "mx_last_error", "mx_status_string", "mx_payload_bytes", "mx_scale_bytes",
    "mx_quantize_workspace_bytes", "mx_quantize", "mx_grouped_gemm", "mx_grouped_gemm_swiglu_fwd",
    "mx_grouped_gemm_dswiglu_bwd", "mx_grouped_gemm_wgrad", "mx_mlp_workspace_bytes", "mx_mlp_fwd_bwd",
    "mx_get_device_status", "mx_selftest_bounded_wait", "mx_gemm_bias", "mx_gemm_gelu_fwd",
    "mx_gemm_dgelu_workspace_bytes", "mx_gemm_dgelu_bwd", "mx_quantize_colsum_noalloc", "mx_debug_tap",
    "mx_mlp_pipeline_create", "mx_mlp_pipeline_run", "mx_mlp_pipeline_sync", "mx_mlp_pipeline_destroy",
    "mx_grouped_gemm_wgrad_f32", "mx_grouped_gemm_swiglu_probs_fwd", "mx_dswiglu_probs_workspace_bytes",
    "mx_grouped_gemm_dswiglu_probs_bwd", "mx_quantize_sr", "mx_moe_route_rows", "mx_moe_route_workspace_bytes",
    "mx_moe_route_index", "mx_permute_quantize", "mx_moe_unpermute", "mx_grouped_gemm_bias", "mx_grouped_gemm_bias_2sm",
    "mx_grouped_gemm_wgrad_workspace_bytes", "mx_grouped_gemm_wgrad_ws", "mx_grouped_gemm_wgrad_f32_ws",
    "mx_mlp_workspace_layout", "mx_moe_route_rows_pad", "mx_moe_route_index_pad", "mx_grouped_gemm_2sm",
)


class MXError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__("%s: %s" % (self.name, message))


class MxTensorStruct(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("fmt", ctypes.c_int32), ("hadamard", ctypes.c_int32)]


class MlpArgsStruct(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32), ("hadamard", ctypes.c_int32),
                ("G", ctypes.c_int32), ("R", ctypes.c_int64), ("D", ctypes.c_int64), ("F", ctypes.c_int64),
                ("offsets", ctypes.c_void_p), ("x", ctypes.c_void_p), ("w1", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("dy", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("y", ctypes.c_void_p), ("dx", ctypes.c_void_p),
                ("dw1", ctypes.c_void_p), ("dw2", ctypes.c_void_p), ("db1", ctypes.c_void_p),
                ("db2", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class MlpSlotStruct(ctypes.Structure):
    _fields_ = [("data", ctypes.c_size_t), ("scale", ctypes.c_size_t), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64)]


MLP_SLOTS = ("x_row", "x_col", "w1_row", "w1t_row", "w2_row", "w2t_row", "h_row", "h_col", "dy_row", "dy_col",
             "dz_row", "dz_col")


class MlpLayoutStruct(ctypes.Structure):
    _fields_ = [(n, MlpSlotStruct) for n in MLP_SLOTS] + [("z", ctypes.c_size_t), ("total", ctypes.c_size_t)]


class HostIOStruct(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "w1", "w2", "dy", "b1", "b2", "offsets", "y", "dx", "dw1",
                                               "dw2", "db1", "db2")]


_lib = None


def load(path=None):
    """Load the CUDA library (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("MX CUDA library not built at %s (run __graft_entry__.build())" % path)
    L = ctypes.CDLL(path)
    vp, i64, i32, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    tp = ctypes.POINTER(MxTensorStruct)
    sig = {
        "mx_abi_version": (ctypes.c_int, []),
        "mx_last_error": (ctypes.c_char_p, []),
        "mx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mx_payload_bytes": (sz, [i64, i64, i32]),
        "mx_scale_bytes": (sz, [i64, i64]),
        "mx_quantize_workspace_bytes": (sz, [i64, i64, u32]),
        "mx_quantize": (ctypes.c_int, [vp, i64, i64, i64, i64, i32, u32, tp, tp, vp, vp, sz, vp]),
        "mx_grouped_gemm": (ctypes.c_int, [tp, tp, i32, vp, vp, i64, vp]),
        "mx_grouped_gemm_2sm": (ctypes.c_int, [tp, tp, i32, vp, vp, i64, vp]),
        "mx_grouped_gemm_swiglu_fwd": (ctypes.c_int, [tp, tp, i32, vp, tp, tp, vp, vp]),
        "mx_grouped_gemm_dswiglu_bwd": (ctypes.c_int, [tp, tp, vp, i32, vp, tp, tp, vp]),
        "mx_grouped_gemm_wgrad": (ctypes.c_int, [tp, tp, i32, vp, vp, vp]),
        "mx_grouped_gemm_wgrad_f32": (ctypes.c_int, [tp, tp, i32, vp, vp, i32, vp]),
        "mx_grouped_gemm_swiglu_probs_fwd": (ctypes.c_int, [tp, tp, i32, vp, vp, tp, tp, vp, vp]),
        "mx_dswiglu_probs_workspace_bytes": (sz, [i64, i64]),
        "mx_grouped_gemm_dswiglu_probs_bwd": (ctypes.c_int, [tp, tp, vp, vp, i32, vp, tp, tp, vp, vp, sz, vp]),
        "mx_mlp_workspace_bytes": (sz, [ctypes.POINTER(MlpArgsStruct)]),
        "mx_mlp_workspace_layout": (ctypes.c_int, [ctypes.POINTER(MlpArgsStruct), ctypes.POINTER(MlpLayoutStruct)]),
        "mx_mlp_fwd_bwd": (ctypes.c_int, [ctypes.POINTER(MlpArgsStruct), vp]),
        "mx_get_device_status": (ctypes.c_int, [vp]),
        "mx_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint64, vp]),
        "mx_gemm_bias": (ctypes.c_int, [tp, tp, vp, vp, i64, vp]),
        "mx_gemm_gelu_fwd": (ctypes.c_int, [tp, tp, vp, vp, tp, tp, vp]),
        "mx_gemm_dgelu_workspace_bytes": (sz, [i64, i64]),
        "mx_gemm_dgelu_bwd": (ctypes.c_int, [tp, tp, vp, tp, tp, vp, vp, sz, vp]),
        "mx_quantize_colsum_noalloc": (ctypes.c_int, [vp, i64, i64, i64, i32, u32, tp, tp, vp, vp]),
        "mx_quantize_sr": (ctypes.c_int, [vp, i64, i64, i64, i64, i32, u32, ctypes.c_uint64, tp, tp, vp]),
        "mx_moe_route_rows": (i64, [i64, i32, i32]),
        "mx_moe_route_workspace_bytes": (sz, [i64, i32, i32]),
        "mx_moe_route_index": (ctypes.c_int, [vp, i64, i32, i32, vp, vp, i64, vp, vp, sz, vp]),
        "mx_moe_route_rows_pad": (i64, [i64, i32, i32, i32]),
        "mx_moe_route_index_pad": (ctypes.c_int, [vp, i64, i32, i32, i32, vp, vp, i64, vp, vp, sz, vp]),
        "mx_permute_quantize": (ctypes.c_int, [vp, i64, i64, i64, vp, i64, vp, i32, i32, u32, tp, tp, vp]),
        "mx_moe_unpermute": (ctypes.c_int, [vp, i64, i64, vp, vp, i64, i32, vp, vp]),
        "mx_grouped_gemm_bias": (ctypes.c_int, [tp, tp, i32, vp, vp, vp, i64, vp]),
        "mx_grouped_gemm_bias_2sm": (ctypes.c_int, [tp, tp, i32, vp, vp, vp, i64, vp]),
        "mx_grouped_gemm_wgrad_workspace_bytes": (sz, [i64, i64, i64, i32]),
        "mx_grouped_gemm_wgrad_ws": (ctypes.c_int, [tp, tp, i32, vp, vp, vp, sz, vp]),
        "mx_grouped_gemm_wgrad_f32_ws": (ctypes.c_int, [tp, tp, i32, vp, vp, i32, vp, sz, vp]),
        "mx_debug_tap": (ctypes.c_int, [vp, i64]),
        "mx_mlp_pipeline_create": (ctypes.c_int, [ctypes.POINTER(MlpArgsStruct), vp, ctypes.POINTER(vp)]),
        "mx_mlp_pipeline_run": (ctypes.c_int, [vp, ctypes.POINTER(HostIOStruct)]),
        "mx_mlp_pipeline_sync": (ctypes.c_int, [vp]),
        "mx_mlp_pipeline_destroy": (None, [vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status):
    if status != 0:
        raise MXError(status, load().mx_last_error().decode())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# --------------------------------------------------------------------------
# Quantized tensors
# --------------------------------------------------------------------------

def payload_bytes(rows, cols, fmt):
    return int(load().mx_payload_bytes(rows, cols, fmt))


def scale_bytes(rows, cols):
    return int(load().mx_scale_bytes(rows, cols))


class MX:
    """A quantized MX tensor [rows, cols] (blocks along cols) in torch buffers."""

    def __init__(self, rows, cols, fmt=E4M3, hadamard=False, device="cuda", data=None, scale=None):
        import torch
        self.rows, self.cols, self.fmt, self.hadamard = int(rows), int(cols), int(fmt), bool(hadamard)
        rb = payload_bytes(1, cols, fmt)
        self.data = data if data is not None else torch.empty((rows, rb), dtype=torch.uint8, device=device)
        self.scale = scale if scale is not None else torch.empty(scale_bytes(rows, cols), dtype=torch.uint8,
                                                                 device=device)

    def struct(self):
        return MxTensorStruct(self.data.data_ptr(), self.scale.data_ptr(), self.rows, self.cols, self.fmt,
                              1 if self.hadamard else 0)


def _s(m):
    return None if m is None else ctypes.byref(m.struct())


# --------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# --------------------------------------------------------------------------

def mx_quantize(x, fmt=E4M3, rowwise=True, colwise=True, hadamard=False, colsum=False, out_row=None,
                out_col=None, colsum_out=None, workspace=None, stream=None):
    """x: BF16 [rows, cols] or [batch, rows, cols] on the GPU.  Returns
    (out_row [batch*rows, cols], out_col [batch*cols, rows], colsum [cols])."""
    import torch
    assert x.dtype == torch.bfloat16
    batch = x.shape[0] if x.dim() == 3 else 1
    rows, cols = x.shape[-2], x.shape[-1]
    ld = x.stride(-2)
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (HADAMARD if hadamard else 0) | \
            (COLSUM if colsum else 0)
    if rowwise and out_row is None:
        out_row = MX(batch * rows, cols, fmt, hadamard, x.device)
    if colwise and out_col is None:
        out_col = MX(batch * cols, rows, fmt, hadamard, x.device)
    ws_bytes = 0
    if colsum:
        if colsum_out is None:
            colsum_out = torch.empty(cols, dtype=torch.float32, device=x.device)
        ws_bytes = int(load().mx_quantize_workspace_bytes(rows, cols, flags))
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().mx_quantize(_ptr(x), batch, rows, cols, ld, fmt, flags, _s(out_row) if rowwise else None,
                              _s(out_col) if colwise else None, _ptr(colsum_out) if colsum else None,
                              _ptr(workspace) if colsum else None, ws_bytes, _stream(stream)))
    return out_row, out_col, colsum_out


def mx_quantize_sr(x, fmt, seed, rowwise=True, colwise=True, hadamard=False, out_row=None, out_col=None,
                   stream=None):
    """mx_quantize with stochastic rounding of the elements (E2M3 / E2M1);
    returns (out_row, out_col)."""
    import torch
    assert x.dtype == torch.bfloat16
    batch = x.shape[0] if x.dim() == 3 else 1
    rows, cols = x.shape[-2], x.shape[-1]
    ld = x.stride(-2)
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (HADAMARD if hadamard else 0)
    if rowwise and out_row is None:
        out_row = MX(batch * rows, cols, fmt, hadamard, x.device)
    if colwise and out_col is None:
        out_col = MX(batch * cols, rows, fmt, hadamard, x.device)
    _check(load().mx_quantize_sr(x.data_ptr(), batch, rows, cols, ld, fmt, flags, int(seed),
                                 _s(out_row) if rowwise else None, _s(out_col) if colwise else None,
                                 _stream(stream)))
    return out_row, out_col


def mx_moe_route_rows(T, k, G):
    return int(load().mx_moe_route_rows(T, k, G))


def mx_moe_route_index(topk, G, R_cap=None, offsets=None, src=None, row_of=None, workspace=None, stream=None,
                       pad=128):
    """topk int32 [T, k] expert ids on the GPU -> (offsets [G], src [R_cap],
    row_of [T, k]) of the token permute; segments padded to `pad` (128 or
    256) rows."""
    import torch
    assert topk.dtype == torch.int32 and topk.is_contiguous()
    T, k = topk.shape
    dev = topk.device
    R_cap = R_cap if R_cap is not None else int(load().mx_moe_route_rows_pad(T, k, G, pad))
    offsets = offsets if offsets is not None else torch.empty(G, dtype=torch.int32, device=dev)
    src = src if src is not None else torch.empty(R_cap, dtype=torch.int32, device=dev)
    row_of = row_of if row_of is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    nbytes = int(load().mx_moe_route_workspace_bytes(T, k, G))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check(load().mx_moe_route_index_pad(_ptr(topk), T, k, G, pad, _ptr(offsets), _ptr(src), R_cap, _ptr(row_of),
                                          _ptr(workspace), workspace.numel(), _stream(stream)))
    return offsets, src, row_of


def mx_permute_quantize(x, src, offsets=None, G=0, fmt=E4M3, rowwise=True, colwise=True, out_row=None,
                        out_col=None, stream=None):
    """The quantizing permute of BF16 tokens x [T, D] by src [R_cap]:
    returns (out_row [R_cap, D], out_col [D, R_cap])."""
    import torch
    assert x.dtype == torch.bfloat16 and src.dtype == torch.int32
    T, D = x.shape
    R_cap = src.numel()
    if offsets is not None and not G:
        G = offsets.numel()
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0)
    if rowwise and out_row is None:
        out_row = MX(R_cap, D, fmt, False, x.device)
    if colwise and out_col is None:
        out_col = MX(D, R_cap, fmt, False, x.device)
    _check(load().mx_permute_quantize(_ptr(x), T, D, x.stride(0), _ptr(src), R_cap, _ptr(offsets), int(G), fmt, flags,
                                      _s(out_row) if rowwise else None, _s(out_col) if colwise else None,
                                      _stream(stream)))
    return out_row, out_col


def mx_moe_unpermute(inp, row_of, weights=None, out=None, stream=None):
    """out[t] = sum_j w[t, j] * inp[row_of[t, j]] in BF16 (fp32 sums)."""
    import torch
    assert inp.dtype == torch.bfloat16 and inp.is_contiguous() and row_of.dtype == torch.int32
    R, D = inp.shape
    T, k = row_of.shape
    if out is None:
        out = torch.empty((T, D), dtype=torch.bfloat16, device=inp.device)
    _check(load().mx_moe_unpermute(_ptr(inp), R, D, _ptr(row_of), _ptr(weights), T, k, _ptr(out), _stream(stream)))
    return out


def mx_quantize_colsum_noalloc(x, fmt=E4M3, rowwise=True, hadamard=False, out_row=None, out_col=None,
                               colsum_out=None, stream=None):
    """Quantize a BF16 [rows, cols] tensor columnwise (and rowwise) with the
    per-column sums, using the library's fixed scratch instead of a
    workspace: for callers that cannot allocate device memory.  Outputs are
    allocated here only when the caller passes none."""
    import torch
    rows, cols = x.shape
    flags = COLWISE | COLSUM | (ROWWISE if rowwise else 0) | (HADAMARD if hadamard else 0)
    if rowwise and out_row is None:
        out_row = MX(rows, cols, fmt, hadamard, x.device)
    if out_col is None:
        out_col = MX(cols, rows, fmt, hadamard, x.device)
    if colsum_out is None:
        colsum_out = torch.empty(cols, dtype=torch.float32, device=x.device)
    _check(load().mx_quantize_colsum_noalloc(_ptr(x), rows, cols, x.stride(0), fmt, flags,
                                             _s(out_row) if rowwise else None, _s(out_col), _ptr(colsum_out),
                                             _stream(stream)))
    return out_row, out_col, colsum_out


def mx_grouped_gemm(a, b, G, offsets, out=None, ld_out=None, stream=None):
    import torch
    N = b.rows // G if G else 0
    if out is None:
        out = torch.empty((a.rows, N), dtype=torch.bfloat16, device=a.data.device)
    ld = ld_out if ld_out is not None else out.stride(0)
    _check(load().mx_grouped_gemm(_s(a), _s(b), G, _ptr(offsets), _ptr(out), ld, _stream(stream)))
    return out


def mx_grouped_gemm_2sm(a, b, G, offsets, out=None, ld_out=None, stream=None):
    """mx_grouped_gemm on CTA pairs (256-row tiles; segments multiples of
    128, a 128-row remainder's upper half computed and not stored)."""
    import torch
    N = b.rows // G if G else 0
    if out is None:
        out = torch.empty((a.rows, N), dtype=torch.bfloat16, device=a.data.device)
    ld = ld_out if ld_out is not None else out.stride(0)
    _check(load().mx_grouped_gemm_2sm(_s(a), _s(b), G, _ptr(offsets), _ptr(out), ld, _stream(stream)))
    return out


def mx_grouped_gemm_bias_2sm(a, b, G, offsets, bias, out=None, ld_out=None, stream=None):
    """mx_grouped_gemm_bias on CTA pairs."""
    import torch
    N = b.rows // G if G else 0
    assert bias.dtype == torch.bfloat16 and bias.is_contiguous()
    if out is None:
        out = torch.empty((a.rows, N), dtype=torch.bfloat16, device=a.data.device)
    ld = ld_out if ld_out is not None else out.stride(0)
    _check(load().mx_grouped_gemm_bias_2sm(_s(a), _s(b), G, _ptr(offsets), _ptr(bias), _ptr(out), ld,
                                           _stream(stream)))
    return out


def mx_grouped_gemm_bias(a, b, G, offsets, bias, out=None, ld_out=None, stream=None):
    """mx_grouped_gemm with expert g's BF16 bias row bias[g] [G, N] added in
    the fp32 accumulator."""
    import torch
    N = b.rows // G if G else 0
    assert bias.dtype == torch.bfloat16 and bias.is_contiguous()
    if out is None:
        out = torch.empty((a.rows, N), dtype=torch.bfloat16, device=a.data.device)
    ld = ld_out if ld_out is not None else out.stride(0)
    _check(load().mx_grouped_gemm_bias(_s(a), _s(b), G, _ptr(offsets), _ptr(bias), _ptr(out), ld, _stream(stream)))
    return out


def mx_grouped_gemm_swiglu_fwd(x_row, w1_row, G, offsets, h_row=None, h_col=None, z=None, stream=None):
    import torch
    R = x_row.rows
    F = w1_row.rows // (2 * G)
    dev = x_row.data.device
    if h_row is None:
        h_row = MX(R, F, E4M3, False, dev)
    if h_col is None:
        h_col = MX(F, R, E4M3, False, dev)
    if z is None:
        z = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
    _check(load().mx_grouped_gemm_swiglu_fwd(_s(x_row), _s(w1_row), G, _ptr(offsets), _s(h_row), _s(h_col),
                                             _ptr(z), _stream(stream)))
    return z, h_row, h_col


def mx_grouped_gemm_swiglu_probs_fwd(x_row, w1_row, G, offsets, probs, h_row=None, h_col=None, z=None, stream=None):
    """FC1 + SwiGLU with each routed row's activation scaled by probs [R] (fp32)."""
    import torch
    R = x_row.rows
    F = w1_row.rows // (2 * G)
    dev = x_row.data.device
    h_row = h_row if h_row is not None else MX(R, F, E4M3, False, dev)
    h_col = h_col if h_col is not None else MX(F, R, E4M3, False, dev)
    z = z if z is not None else torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
    _check(load().mx_grouped_gemm_swiglu_probs_fwd(_s(x_row), _s(w1_row), G, _ptr(offsets), _ptr(probs), _s(h_row),
                                                   _s(h_col), _ptr(z), _stream(stream)))
    return z, h_row, h_col


def mx_grouped_gemm_dswiglu_probs_bwd(dy_row, w2t_row, z, probs, G, offsets, dz_row=None, dz_col=None,
                                      dprobs=None, workspace=None, stream=None):
    """The matching backward; returns (dz_row, dz_col, dprobs [R] fp32)."""
    import torch
    R = dy_row.rows
    F = w2t_row.rows // G
    dev = dy_row.data.device
    dz_row = dz_row if dz_row is not None else MX(R, 2 * F, E4M3, False, dev)
    dz_col = dz_col if dz_col is not None else MX(2 * F, R, E4M3, False, dev)
    dprobs = dprobs if dprobs is not None else torch.empty(R, dtype=torch.float32, device=dev)
    nbytes = int(load().mx_dswiglu_probs_workspace_bytes(R, F))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check(load().mx_grouped_gemm_dswiglu_probs_bwd(
        _s(dy_row), _s(w2t_row), _ptr(z), _ptr(probs), G, _ptr(offsets), _s(dz_row), _s(dz_col), _ptr(dprobs),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return dz_row, dz_col, dprobs


def mx_grouped_gemm_dswiglu_bwd(dy_row, w2t_row, z, G, offsets, dz_row=None, dz_col=None, stream=None):
    R = dy_row.rows
    F = w2t_row.rows // G
    dev = dy_row.data.device
    if dz_row is None:
        dz_row = MX(R, 2 * F, E4M3, False, dev)
    if dz_col is None:
        dz_col = MX(2 * F, R, E4M3, False, dev)
    _check(load().mx_grouped_gemm_dswiglu_bwd(_s(dy_row), _s(w2t_row), _ptr(z), G, _ptr(offsets), _s(dz_row),
                                              _s(dz_col), _stream(stream)))
    return dz_row, dz_col


def mx_grouped_gemm_wgrad(a_col, b_col, G, offsets, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((G, a_col.rows, b_col.rows), dtype=torch.bfloat16, device=a_col.data.device)
    _check(load().mx_grouped_gemm_wgrad(_s(a_col), _s(b_col), G, _ptr(offsets), _ptr(out), _stream(stream)))
    return out


def mx_grouped_gemm_wgrad_f32(a_col, b_col, G, offsets, grad, accumulate=False, stream=None):
    """Weight gradient into the caller's fp32 buffer grad [G, N, K]: stored
    (accumulate=False) or added to what it holds (accumulate=True)."""
    import torch
    assert grad.dtype == torch.float32 and grad.is_contiguous()
    _check(load().mx_grouped_gemm_wgrad_f32(_s(a_col), _s(b_col), G, _ptr(offsets), _ptr(grad),
                                            1 if accumulate else 0, _stream(stream)))
    return grad


def mx_grouped_gemm_wgrad_workspace_bytes(N, K, R, G):
    return int(load().mx_grouped_gemm_wgrad_workspace_bytes(N, K, R, G))


def _wgrad_ws(a_col, b_col, G, workspace):
    import torch
    if workspace is None:
        n = mx_grouped_gemm_wgrad_workspace_bytes(a_col.rows, b_col.rows, a_col.cols, G)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=a_col.data.device)
    return workspace


def mx_grouped_gemm_wgrad_ws(a_col, b_col, G, offsets, out=None, workspace=None, stream=None):
    """mx_grouped_gemm_wgrad with the largest experts' K range split across
    CTAs (workspace from mx_grouped_gemm_wgrad_workspace_bytes)."""
    import torch
    if out is None:
        out = torch.empty((G, a_col.rows, b_col.rows), dtype=torch.bfloat16, device=a_col.data.device)
    ws = _wgrad_ws(a_col, b_col, G, workspace)
    _check(load().mx_grouped_gemm_wgrad_ws(_s(a_col), _s(b_col), G, _ptr(offsets), _ptr(out), _ptr(ws), ws.numel(),
                                           _stream(stream)))
    return out


def mx_grouped_gemm_wgrad_f32_ws(a_col, b_col, G, offsets, grad, accumulate=False, workspace=None, stream=None):
    import torch
    assert grad.dtype == torch.float32 and grad.is_contiguous()
    ws = _wgrad_ws(a_col, b_col, G, workspace)
    _check(load().mx_grouped_gemm_wgrad_f32_ws(_s(a_col), _s(b_col), G, _ptr(offsets), _ptr(grad),
                                               1 if accumulate else 0, _ptr(ws), ws.numel(), _stream(stream)))
    return grad


def mx_gemm_bias(a, b, bias=None, out=None, ld_out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.data.device)
    ld = ld_out if ld_out is not None else out.stride(0)
    _check(load().mx_gemm_bias(_s(a), _s(b), _ptr(bias), _ptr(out), ld, _stream(stream)))
    return out


def mx_gemm_gelu_fwd(x_row, w1_row, b1=None, pre=None, act_row=None, act_col=None, fmt=E2M3, hadamard=True,
                     stream=None):
    import torch
    M, H = x_row.rows, w1_row.rows
    dev = x_row.data.device
    if pre is None:
        pre = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    if act_row is None:
        act_row = MX(M, H, fmt, hadamard, dev)
    if act_col is None:
        act_col = MX(H, M, fmt, hadamard, dev)
    _check(load().mx_gemm_gelu_fwd(_s(x_row), _s(w1_row), _ptr(b1), _ptr(pre), _s(act_row), _s(act_col),
                                   _stream(stream)))
    return pre, act_row, act_col


def mx_gemm_dgelu_workspace_bytes(M, H):
    return int(load().mx_gemm_dgelu_workspace_bytes(M, H))


def mx_gemm_dgelu_bwd(dy_row, w2t_row, pre, dpre_row=None, dpre_col=None, db1=None, workspace=None, fmt=E2M3,
                      hadamard=True, stream=None):
    import torch
    M, H = dy_row.rows, w2t_row.rows
    dev = dy_row.data.device
    if dpre_row is None:
        dpre_row = MX(M, H, fmt, hadamard, dev)
    if dpre_col is None:
        dpre_col = MX(H, M, fmt, hadamard, dev)
    if db1 is None:
        db1 = torch.empty(H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(mx_gemm_dgelu_workspace_bytes(M, H), 16), dtype=torch.uint8, device=dev)
    _check(load().mx_gemm_dgelu_bwd(_s(dy_row), _s(w2t_row), _ptr(pre), _s(dpre_row), _s(dpre_col), _ptr(db1),
                                    _ptr(workspace), workspace.numel(), _stream(stream)))
    return dpre_row, dpre_col, db1


def mlp_args(x, w1, w2, dy, offsets, G, F, y, dx, dw1, dw2, workspace=None, act=ACT_SWIGLU, fmt=E4M3,
             hadamard=False, b1=None, b2=None, db1=None, db2=None):
    R, D = x.shape
    a = MlpArgsStruct()
    a.act, a.fmt, a.hadamard, a.G = act, fmt, 1 if hadamard else 0, G
    a.R, a.D, a.F = R, D, F
    for name, t in (("offsets", offsets), ("x", x), ("w1", w1), ("w2", w2), ("dy", dy), ("b1", b1), ("b2", b2),
                    ("y", y), ("dx", dx), ("dw1", dw1), ("dw2", dw2), ("db1", db1), ("db2", db2)):
        setattr(a, name, None if t is None else t.data_ptr())
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def mx_mlp_workspace_bytes(args):
    return int(load().mx_mlp_workspace_bytes(ctypes.byref(args)))


def mx_mlp_workspace_layout(args):
    """{slot: (payload offset, scale offset, rows, cols)} for every quantized
    tensor of the step, plus "z" (offset of the BF16 pre-activation) and
    "total" (workspace bytes)."""
    out = MlpLayoutStruct()
    _check(load().mx_mlp_workspace_layout(ctypes.byref(args), ctypes.byref(out)))
    lay = {n: (int(getattr(out, n).data), int(getattr(out, n).scale), int(getattr(out, n).rows),
               int(getattr(out, n).cols)) for n in MLP_SLOTS}
    lay["z"] = int(out.z)
    lay["total"] = int(out.total)
    return lay


def mlp_workspace_views(args, workspace):
    """The step's intermediates as views into its workspace (uint8 torch
    tensor): {slot: MX} and "z" (BF16 [R, F1])."""
    import torch
    lay = mx_mlp_workspace_layout(args)
    views = {}
    for n in MLP_SLOTS:
        d, sc, rows, cols = lay[n]
        rb = payload_bytes(1, cols, args.fmt)
        data = workspace[d:d + rows * rb].view(rows, rb)
        scale = workspace[sc:sc + scale_bytes(rows, cols)]
        views[n] = MX(rows, cols, args.fmt, bool(args.hadamard), workspace.device, data=data, scale=scale)
    f1 = lay["dz_row"][3]
    views["z"] = workspace[lay["z"]:lay["z"] + args.R * f1 * 2].view(torch.bfloat16).view(args.R, f1)
    return views


def mx_mlp_fwd_bwd(args, stream=None):
    _check(load().mx_mlp_fwd_bwd(ctypes.byref(args), _stream(stream)))


class MlpPipeline:
    """The step with host-memory inputs and outputs (mx_mlp_pipeline_*).

    dev_args: the device argument block (mlp_args with a workspace) whose
    buffers the pipeline stages through; the tensors behind it must outlive
    the pipeline.  run(host) takes CPU tensors (pinned, for overlap) keyed
    x, w1, w2, dy, offsets, y, dx, dw1, dw2 (and b1, b2, db1, db2 for GELU);
    they are read and written asynchronously until sync()."""

    def __init__(self, dev_args, stream=None):
        self._args = dev_args
        h = ctypes.c_void_p()
        _check(load().mx_mlp_pipeline_create(ctypes.byref(dev_args), _stream(stream), ctypes.byref(h)))
        self._h = h
        self._io = []

    def run(self, host):
        io = HostIOStruct()
        for name, _ in HostIOStruct._fields_:
            t = host.get(name)
            setattr(io, name, None if t is None else t.data_ptr())
        self._io.append(io)
        _check(load().mx_mlp_pipeline_run(self._h, ctypes.byref(io)))

    def sync(self):
        _check(load().mx_mlp_pipeline_sync(self._h))
        self._io = []

    def close(self):
        if self._h is not None:
            load().mx_mlp_pipeline_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mx_get_device_status(stream=None):
    """Synchronise and return the device status name ('MX_OK' or an error)."""
    return STATUS.get(int(load().mx_get_device_status(_stream(stream))), "unknown")


def mx_selftest_bounded_wait(budget_ns, stream=None):
    _check(load().mx_selftest_bounded_wait(int(budget_ns), _stream(stream)))


def mx_debug_tap(tap=None):
    """Attach (fp32 CUDA tensor) or detach (None) the fused epilogues' test
    tap on this host thread: they also write their fp32 pre-quantization
    values into it, row-major [rows, cols] of the requantized output."""
    if tap is None:
        _check(load().mx_debug_tap(None, 0))
        return
    import torch
    assert tap.dtype == torch.float32 and tap.is_cuda and tap.is_contiguous()
    _check(load().mx_debug_tap(tap.data_ptr(), tap.numel()))


def mx_last_error():
    return load().mx_last_error().decode()
