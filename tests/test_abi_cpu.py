"""The C ABI on the host: the library builds, loads and exports every symbol
include/mx.h declares; malformed calls are rejected by the host validation
before any device work (no GPU needed: rejected calls never reach CUDA).
Pointers passed here are never dereferenced."""
import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mx():
    from mlp_gemms_gb300 import build
    build.build()
    import mlp_gemms_gb300 as m
    m.load()
    return m


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mx.h")).read()
    return sorted(set(re.findall(r"^MX_API [^;]*?\b(mx_\w+)\(", src, flags=re.M)))


def test_exports_every_declared_symbol(mx):
    decl = declared_symbols()
    assert len(decl) >= 15
    lib = mx.load()
    for name in decl:
        assert hasattr(lib, name), name
    assert sorted(mx.ABI_SYMBOLS) == decl
    assert lib.mx_abi_version() == 1


def test_sizes_agree_with_the_oracle(mx):
    for rows, cols, fmt in [(256, 256, 0), (96, 160, 1), (1000, 4096, 2), (7168, 8192, 0)]:
        assert mx.payload_bytes(rows, cols, fmt) == rows * O.payload_row_bytes(cols, fmt)
        assert mx.scale_bytes(rows, cols) == O.scale_bytes(rows, cols // 32)


FAKE = 0x10000          # 16-byte aligned, never dereferenced
MISALIGNED = 0x10008


def _t(rows, cols, fmt=0, had=0, data=FAKE, scale=FAKE):
    from mlp_gemms_gb300 import MxTensorStruct
    return MxTensorStruct(data, scale, rows, cols, fmt, had)


def _quant(mx, **kw):
    a = dict(x=FAKE, batch=1, rows=256, cols=256, ld=256, fmt=0, flags=3, out_row=_t(256, 256),
             out_col=_t(256, 256), colsum=None, ws=None, ws_bytes=0)
    a.update(kw)
    st = mx.load().mx_quantize(a["x"], a["batch"], a["rows"], a["cols"], a["ld"], a["fmt"], a["flags"],
                               ctypes.byref(a["out_row"]) if a["out_row"] is not None else None,
                               ctypes.byref(a["out_col"]) if a["out_col"] is not None else None,
                               a["colsum"], a["ws"], a["ws_bytes"], None)
    return mx.STATUS[st], mx.mx_last_error()


@pytest.mark.parametrize("kw,status,word", [
    (dict(fmt=7), "MX_ERR_INVALID_ARG", "fmt"),
    (dict(flags=0), "MX_ERR_INVALID_ARG", "MX_ROWWISE"),
    (dict(flags=0x30), "MX_ERR_INVALID_ARG", "flag"),
    (dict(cols=250, ld=256), "MX_ERR_SHAPE", "cols"),
    (dict(rows=100), "MX_ERR_SHAPE", "rows"),
    (dict(ld=200), "MX_ERR_ALIGNMENT", "ld"),
    (dict(x=MISALIGNED), "MX_ERR_ALIGNMENT", "x"),
    (dict(x=None), "MX_ERR_INVALID_ARG", "x"),
    (dict(batch=0), "MX_ERR_SHAPE", "batch"),
    (dict(batch=2, rows=96, out_row=None, out_col=None, flags=1), "MX_ERR_SHAPE", "batched"),
    (dict(out_row=None), "MX_ERR_INVALID_ARG", "out_row"),
    (dict(out_col=None), "MX_ERR_INVALID_ARG", "out_col"),
    # sizes whose element products would overflow 64 bits if multiplied unchecked
    (dict(rows=1 << 62, ld=1 << 40, flags=1), "MX_ERR_SHAPE", "too large"),
    (dict(rows=1 << 30, ld=1 << 39, batch=1 << 30, flags=1), "MX_ERR_SHAPE", "too large"),
    (dict(rows=1 << 20, ld=1 << 21, flags=1), "MX_ERR_SHAPE", "too large"),
], ids=lambda v: str(v))
def test_quantize_rejections(mx, kw, status, word):
    if kw.get("out_row", 1) is None and "flags" in kw:
        pass
    st, msg = _quant(mx, **kw)
    assert st == status, msg
    assert word in msg


def test_quantize_tensor_mismatches(mx):
    st, msg = _quant(mx, out_row=_t(256, 128))
    assert st == "MX_ERR_SHAPE" and "out_row" in msg
    st, msg = _quant(mx, out_row=_t(256, 256, fmt=1))
    assert st == "MX_ERR_INVALID_ARG" and "format" in msg
    st, msg = _quant(mx, out_col=_t(256, 256, had=1))
    assert st == "MX_ERR_INVALID_ARG" and "rotation" in msg
    st, msg = _quant(mx, out_row=_t(256, 256, data=MISALIGNED))
    assert st == "MX_ERR_ALIGNMENT"
    st, msg = _quant(mx, flags=3 | 8)
    assert st == "MX_ERR_INVALID_ARG" and "colsum" in msg
    st, msg = _quant(mx, flags=1 | 8, out_col=None, colsum=FAKE)
    assert st == "MX_ERR_INVALID_ARG" and "MX_COLWISE" in msg
    st, msg = _quant(mx, flags=3 | 8, colsum=FAKE, ws=FAKE, ws_bytes=16)
    assert st == "MX_ERR_WORKSPACE"


def _gemm(mx, a, b, G=1, offsets=FAKE, out=FAKE, ld=None):
    ld = ld if ld is not None else (b.rows // max(G, 1))
    st = mx.load().mx_grouped_gemm(ctypes.byref(a), ctypes.byref(b), G, offsets, out, ld, None)
    return mx.STATUS[st], mx.mx_last_error()


def test_grouped_gemm_rejections(mx):
    assert _gemm(mx, _t(256, 256), _t(256, 256), G=0)[0] == "MX_ERR_INVALID_ARG"
    assert _gemm(mx, _t(256, 256), _t(256, 192))[0] == "MX_ERR_SHAPE"          # K mismatch
    assert _gemm(mx, _t(256, 192), _t(256, 192))[0] == "MX_ERR_SHAPE"          # K % 128
    assert _gemm(mx, _t(256, 256), _t(384, 256), G=2)[0] == "MX_ERR_SHAPE"     # N = 192
    assert _gemm(mx, _t(256, 256, fmt=1), _t(256, 256, fmt=0))[0] == "MX_ERR_INVALID_ARG"   # mixed formats
    assert _gemm(mx, _t(256, 256, had=1), _t(256, 256))[0] == "MX_ERR_INVALID_ARG"          # rotation on one side
    assert _gemm(mx, _t(256, 256, fmt=1, data=FAKE + 16), _t(256, 256, fmt=1))[0] == "MX_ERR_ALIGNMENT"
    assert _gemm(mx, _t(256, 256, fmt=5), _t(256, 256, fmt=5))[0] == "MX_ERR_INVALID_ARG"
    assert _gemm(mx, _t(256, 256), _t(256, 256), out=MISALIGNED)[0] == "MX_ERR_ALIGNMENT"
    assert _gemm(mx, _t(256, 256), _t(256, 256), ld=100)[0] == "MX_ERR_ALIGNMENT"
    assert _gemm(mx, _t(256, 256), _t(512, 256), G=2, offsets=None)[0] == "MX_ERR_INVALID_ARG"
    assert _gemm(mx, _t(256, 256, data=MISALIGNED), _t(256, 256))[0] == "MX_ERR_ALIGNMENT"


def test_fused_and_wgrad_rejections(mx):
    L = mx.load()
    x, w1 = _t(1024, 256), _t(2 * 2 * 256, 256)
    h_row, h_col = _t(1024, 256), _t(256, 1024)
    st = L.mx_grouped_gemm_swiglu_fwd(ctypes.byref(x), ctypes.byref(w1), 2, FAKE, ctypes.byref(_t(1024, 128)),
                                      ctypes.byref(h_col), FAKE, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE" and "h_row" in mx.mx_last_error()
    st = L.mx_grouped_gemm_swiglu_fwd(ctypes.byref(x), ctypes.byref(_t(3 * 256, 256)), 2, FAKE,
                                      ctypes.byref(h_row), ctypes.byref(h_col), FAKE, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE"
    st = L.mx_grouped_gemm_swiglu_fwd(ctypes.byref(_t(1000, 256)), ctypes.byref(w1), 2, FAKE,
                                      ctypes.byref(h_row), ctypes.byref(h_col), FAKE, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE"
    dy, w2t = _t(1024, 256), _t(2 * 256, 256)
    st = L.mx_grouped_gemm_dswiglu_bwd(ctypes.byref(dy), ctypes.byref(w2t), FAKE, 2, FAKE,
                                       ctypes.byref(_t(1024, 512)), ctypes.byref(_t(512, 1000)), None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE" and "dz_col" in mx.mx_last_error()
    st = L.mx_grouped_gemm_wgrad(ctypes.byref(_t(256, 1024)), ctypes.byref(_t(384, 1000)), 2, FAKE, FAKE, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE"
    st = L.mx_grouped_gemm_wgrad(ctypes.byref(_t(256, 1024)), ctypes.byref(_t(384, 1024)), 0, FAKE, FAKE, None)
    assert mx.STATUS[st] == "MX_ERR_INVALID_ARG"


def test_mlp_rejections_and_workspace_size(mx):
    a = mx.MlpArgsStruct()
    a.act, a.fmt, a.G, a.R, a.D, a.F = 0, 0, 128, 262144, 2048, 768
    ws = mx.mx_mlp_workspace_bytes(a)
    # every quantized operand of the step plus the BF16 pre-activation
    R, D, F, G = 262144, 2048, 768, 128
    payload = 2 * R * D + 6 * G * D * F + 2 * R * F + 2 * R * D + 4 * R * F + 4 * R * F
    # plus the wgrad K-split workspace, shared by dW2 [D, F] and dW1 [2F, D]
    split = max(mx.mx_grouped_gemm_wgrad_workspace_bytes(D, F, R, G),
                mx.mx_grouped_gemm_wgrad_workspace_bytes(2 * F, D, R, G))
    assert 0 < split < 0.1 * payload
    assert payload + split < ws < (payload + split) * 1.05
    st = mx.load().mx_mlp_fwd_bwd(ctypes.byref(a), None)
    assert mx.STATUS[st] == "MX_ERR_INVALID_ARG"          # NULL tensors
    a.act = 1
    st = mx.load().mx_mlp_fwd_bwd(ctypes.byref(a), None)
    assert mx.STATUS[st] == "MX_ERR_NOT_SUPPORTED"


@pytest.mark.parametrize("act,fmt,G,R,D,F", [(0, 0, 128, 262144, 2048, 768), (0, 0, 2, 512, 256, 128),
                                             (1, 1, 1, 16384, 3072, 12288)])
def test_mlp_workspace_layout(mx, act, fmt, G, R, D, F):
    """The step's workspace layout: every slot sized for its tensor's payload
    and blocked scales, all slots and the BF16 pre-activation disjoint and
    16-byte aligned, inside mx_mlp_workspace_bytes."""
    a = mx.MlpArgsStruct()
    a.act, a.fmt, a.G, a.R, a.D, a.F = act, fmt, G, R, D, F
    lay = mx.mx_mlp_workspace_layout(a)
    assert lay["total"] == mx.mx_mlp_workspace_bytes(a)
    F1 = 2 * F if act == 0 else F
    shapes = {"x_row": (R, D), "x_col": (D, R), "w1_row": (G * F1, D), "w1t_row": (G * D, F1),
              "w2_row": (G * D, F), "w2t_row": (G * F, D), "h_row": (R, F), "h_col": (F, R), "dy_row": (R, D),
              "dy_col": (D, R), "dz_row": (R, F1), "dz_col": (F1, R)}
    spans = []
    for n, (rows, cols) in shapes.items():
        d, sc, r, c = lay[n]
        assert (r, c) == (rows, cols), n
        spans.append((d, d + rows * mx.payload_bytes(1, cols, fmt), n))
        spans.append((sc, sc + mx.scale_bytes(rows, cols), n + " scales"))
    spans.append((lay["z"], lay["z"] + R * F1 * 2, "z"))
    spans.sort()
    for (s0, e0, n0), (s1, e1, n1) in zip(spans, spans[1:]):
        assert e0 <= s1, (n0, n1)
    assert all(s % 16 == 0 for s, _, _ in spans) and spans[-1][1] <= lay["total"]
    bad = mx.MlpArgsStruct()
    with pytest.raises(mx.MXError) as e:
        mx.mx_mlp_workspace_layout(bad)
    assert e.value.name == "MX_ERR_INVALID_ARG"


def test_noalloc_rejects_overflowing_sizes_before_any_device_call(mx):
    """ceil(rows/128) * cols must not wrap past the scratch limit: huge rows
    or cols are refused on their own."""
    L = mx.load()
    for rows, cols in ((1 << 62, 32), (128, 1 << 62), ((1 << 63) - 1, 1 << 40)):
        st = L.mx_quantize_colsum_noalloc(FAKE, rows, cols, cols, 0, 2 | 8, None, ctypes.byref(_t(cols, rows)),
                                          FAKE, None)
        assert mx.STATUS[st] == "MX_ERR_WORKSPACE", (rows, cols)
        assert "scratch" in mx.mx_last_error()


def test_pair_gemm_rejections(mx):
    """mx_grouped_gemm_2sm: host checks before any device work."""
    L = mx.load()
    a, b = _t(512, 256), _t(384, 256)
    st = L.mx_grouped_gemm_2sm(ctypes.byref(a), ctypes.byref(b), 1, FAKE, FAKE, 384, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE" and "256" in mx.mx_last_error()
    a4, b4 = _t(512, 256, fmt=2), _t(512, 256)   # packed E2M1 against E4M3: .kind::mxf4 takes E2M1 on both
    st = L.mx_grouped_gemm_2sm(ctypes.byref(a4), ctypes.byref(b4), 1, FAKE, FAKE, 512, None)
    assert mx.STATUS[st] == "MX_ERR_INVALID_ARG" and "different formats" in mx.mx_last_error()
    a3, b3 = _t(320, 256), _t(256, 256)
    st = L.mx_grouped_gemm_2sm(ctypes.byref(a3), ctypes.byref(b3), 1, None, FAKE, 256, None)
    assert mx.STATUS[st] == "MX_ERR_SHAPE" and "multiple of 128" in mx.mx_last_error()
    a5, b5 = _t(512, 256), _t(1025 * 256, 256)
    st = L.mx_grouped_gemm_2sm(ctypes.byref(a5), ctypes.byref(b5), 1025, FAKE, FAKE, 256, None)
    assert mx.STATUS[st] == "MX_ERR_NOT_SUPPORTED" and "1024" in mx.mx_last_error()
    # the pair bias form: a bias is required, 16-byte aligned, and at least one expert
    st = L.mx_grouped_gemm_bias_2sm(ctypes.byref(_t(512, 256)), ctypes.byref(_t(512, 256)), 1, FAKE, None, FAKE,
                                    512, None)
    assert mx.STATUS[st] == "MX_ERR_ALIGNMENT" and "bias" in mx.mx_last_error()
    st = L.mx_grouped_gemm_bias_2sm(ctypes.byref(_t(512, 256)), ctypes.byref(_t(512, 256)), 1, FAKE, FAKE + 8, FAKE,
                                    512, None)
    assert mx.STATUS[st] == "MX_ERR_ALIGNMENT"
    st = L.mx_grouped_gemm_bias_2sm(ctypes.byref(_t(512, 256)), ctypes.byref(_t(512, 256)), 0, FAKE, FAKE, FAKE,
                                    512, None)
    assert mx.STATUS[st] == "MX_ERR_INVALID_ARG"
    assert L.mx_moe_route_rows_pad(100, 8, 4, 256) == (800 + 255 * 4 + 255) // 256 * 256
    assert L.mx_moe_route_rows_pad(100, 8, 4, 200) == 0
