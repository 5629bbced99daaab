"""Element-wise parity of the whole training step (mx_mlp_fwd_bwd).

The step's quantized intermediates stay in the caller's workspace
(mx_mlp_workspace_layout says where).  After one step the tests read them
back and hold every stage to the oracle on exactly the operands the stage
consumed, as the tolerance rule of the torchao PR #5 page's hardening
commit asks (reference = the oracle on the GPU's own quantized upstream
operands, so one near-tie upstream cannot compound):

* quantizer outputs (X, W1, W2, dY, both orientations): bit-exact with the
  oracle's quantization of the BF16 inputs;
* fused requant outputs (h or the GELU activation, dz or dpre): the stage
  re-run on the chain's own operands with the debug tap attached gives the
  chain's bytes bit for bit, the oracle's quantization of the tapped fp32
  values gives them too, and the tapped values are within tolerance of the
  oracle's;
* float outputs (z / pre, y, dX, dW1, dW2, db1, db2): element by element
  within 2^-8 |ref| + 2^-14 rms(ref row) of the oracle stage.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, assert_tap_requant_exact, bf16_cpu, mx_bytes, to_dev, with_tap

pytestmark = pytest.mark.gpu


def _deq(m, fmt):
    p, s = mx_bytes(m)
    return O.dequantize_rows(p, s, m.rows, m.cols, fmt)


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _close(got, ref, what):
    ok = O.within_tolerance(got, ref)
    assert ok.all(), "%s: %d of %d outside tolerance, first at %s (gpu %r, oracle %r)" % (
        what, int((~ok).sum()), ok.size, np.argwhere(~ok)[0], got[tuple(np.argwhere(~ok)[0])],
        ref[tuple(np.argwhere(~ok)[0])])


def _offsets(counts):
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


@pytest.mark.parametrize("F", [384, 512])
def test_swiglu_step_elementwise(cuda_lib, F):
    """Four experts (one empty) and a 128-row inactive tail; F = 384 runs
    the dSwiGLU epilogue on 128-column tiles, F = 512 on 256-column ones."""
    import torch
    mx = cuda_lib
    G, D, R = 4, 1024, 1152
    offsets = _offsets([384, 0, 256, 384])
    A = int(offsets[-1])
    inp = W.moe_inputs(G, D, F, R, seed=21)
    t = {k: to_dev(v) for k, v in inp.items()}
    out = {"y": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda"),
           "dx": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda"),
           "dw1": torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device="cuda"),
           "dw2": torch.empty((G, D, F), dtype=torch.bfloat16, device="cuda")}
    offs = torch.from_numpy(offsets).cuda()
    a0 = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"], out["dw2"])
    ws = torch.zeros(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device="cuda")
    args = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                       out["dw2"], workspace=ws)
    mx.mx_mlp_fwd_bwd(args)
    assert mx.mx_get_device_status() == "MX_OK"
    V = mx.mlp_workspace_views(args, ws)
    E = O.E4M3

    # quantizers: bit-exact
    xq = O.quantize_bf16(inp["x"], E)
    assert_quant_equal(V["x_row"], (xq["row_payload"], xq["row_scales"]), R, D // 32, "x_row")
    assert_quant_equal(V["x_col"], (xq["col_payload"], xq["col_scales"]), D, R // 32, "x_col")
    assert_quant_equal(V["w1_row"], O.quantize_experts_rows(inp["w1"], E), G * 2 * F, D // 32, "w1_row")
    assert_quant_equal(V["w1t_row"], O.quantize_experts_cols(inp["w1"], E), G * D, 2 * F // 32, "w1t_row")
    assert_quant_equal(V["w2_row"], O.quantize_experts_rows(inp["w2"], E), G * D, F // 32, "w2_row")
    assert_quant_equal(V["w2t_row"], O.quantize_experts_cols(inp["w2"], E), G * F, D // 32, "w2t_row")
    dyq = O.quantize_bf16(inp["dy"], E)
    assert_quant_equal(V["dy_row"], (dyq["row_payload"], dyq["row_scales"]), R, D // 32, "dy_row")
    assert_quant_equal(V["dy_col"], (dyq["col_payload"], dyq["col_scales"]), D, R // 32, "dy_col")

    # FC1 + SwiGLU on the chain's own X and W1
    fwd = O.swiglu_fwd(_deq(V["x_row"], E), _deq(V["w1_row"], E).reshape(G, 2 * F, D), offsets)
    z_bits = _bits(V["z"])
    _close(O.bf16_to_f64(z_bits[:A]), fwd["z"][:A], "z")
    (z2, h2r, h2c), tap = with_tap(mx, R, F, lambda: mx.mx_grouped_gemm_swiglu_fwd(V["x_row"], V["w1_row"], G, offs))
    assert torch.equal(z2[:A], V["z"][:A]), "z differs between the step and the stage"
    assert torch.equal(h2r.data[:A], V["h_row"].data[:A]), "h rowwise differs between the step and the stage"
    assert np.array_equal(mx_bytes(h2c)[0][:, :A], mx_bytes(V["h_col"])[0][:, :A]), \
        "h columnwise differs between the step and the stage"
    assert_tap_requant_exact(V["h_row"], V["h_col"], tap, A, F, R, what="h")
    _close(tap[:A].astype(np.float64), fwd["h"], "h (fp32 before the requant)")

    # FC2 on the chain's own h and W2
    hq = np.concatenate([_deq(V["h_row"], E)[:A], np.zeros((R - A, F))])
    y_ref = O.grouped_gemm(hq, _deq(V["w2_row"], E).reshape(G, D, F), offsets)
    got_y = bf16_cpu(out["y"])
    _close(got_y[:A], y_ref[:A], "y")
    assert np.all(np.isnan(got_y[A:])), "inactive tail of y was written"

    # FC2 dgrad + dSwiGLU on the chain's own dY, W2^T and saved z
    bwd = O.dswiglu_bwd(_deq(V["dy_row"], E), _deq(V["w2t_row"], E).reshape(G, F, D), z_bits, offsets)
    (d2r, d2c), tap = with_tap(mx, R, 2 * F,
                               lambda: mx.mx_grouped_gemm_dswiglu_bwd(V["dy_row"], V["w2t_row"], V["z"], G, offs))
    assert torch.equal(d2r.data[:A], V["dz_row"].data[:A]), "dz rowwise differs between step and stage"
    assert np.array_equal(mx_bytes(d2c)[0][:, :A], mx_bytes(V["dz_col"])[0][:, :A]), \
        "dz columnwise differs between step and stage"
    assert_tap_requant_exact(V["dz_row"], V["dz_col"], tap, A, 2 * F, R, what="dz")
    _close(tap[:A].astype(np.float64), bwd["dz"], "dz (fp32 before the requant)")

    # FC1 dgrad on the chain's own dz and W1^T
    dzq = np.concatenate([_deq(V["dz_row"], E)[:A], np.zeros((R - A, 2 * F))])
    dx_ref = O.grouped_gemm(dzq, _deq(V["w1t_row"], E).reshape(G, D, 2 * F), offsets)
    got_dx = bf16_cpu(out["dx"])
    _close(got_dx[:A], dx_ref[:A], "dx")
    assert np.all(np.isnan(got_dx[A:])), "inactive tail of dx was written"

    # weight gradients on the chain's own columnwise operands
    dw2_ref = O.wgrad(_deq(V["dy_col"], E), _deq(V["h_col"], E), offsets)
    dw1_ref = O.wgrad(_deq(V["dz_col"], E), _deq(V["x_col"], E), offsets)
    _close(bf16_cpu(out["dw2"]), dw2_ref, "dw2")
    _close(bf16_cpu(out["dw1"]), dw1_ref, "dw1")
    assert bool((out["dw1"][1] == 0).all()) and bool((out["dw2"][1] == 0).all()), "empty expert"


@pytest.mark.parametrize("H", [384, 512])
def test_gelu_step_elementwise(cuda_lib, H):
    """The dense MXFP6 + Hadamard + tanh-GELU step; H = 384 runs the GELU
    epilogues on 128-column tiles, H = 512 on 256-column ones."""
    import torch
    mx = cuda_lib
    M, D = 512, 384
    fmt = O.E2M3
    inp = W.dense_inputs(M, D, H, seed=23)
    t = {k: to_dev(v) for k, v in inp.items()}
    out = {"y": torch.empty((M, D), dtype=torch.bfloat16, device="cuda"),
           "dx": torch.empty((M, D), dtype=torch.bfloat16, device="cuda"),
           "dw1": torch.empty((H, D), dtype=torch.bfloat16, device="cuda"),
           "dw2": torch.empty((D, H), dtype=torch.bfloat16, device="cuda"),
           "db1": torch.empty(H, dtype=torch.float32, device="cuda"),
           "db2": torch.empty(D, dtype=torch.float32, device="cuda")}
    kw = dict(act=mx.ACT_GELU_TANH, fmt=fmt, hadamard=True, b1=t["b1"], b2=t["b2"], db1=out["db1"],
              db2=out["db2"])
    a0 = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], None, 1, H, out["y"], out["dx"], out["dw1"], out["dw2"],
                     **kw)
    ws = torch.zeros(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device="cuda")
    args = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], None, 1, H, out["y"], out["dx"], out["dw1"], out["dw2"],
                       workspace=ws, **kw)
    mx.mx_mlp_fwd_bwd(args)
    assert mx.mx_get_device_status() == "MX_OK"
    V = mx.mlp_workspace_views(args, ws)
    b1 = O.bf16_to_f64(inp["b1"])
    b2 = O.bf16_to_f64(inp["b2"])

    # quantizers (rotated E2M3): bit-exact
    for name, bits, rows, cols in (("x", inp["x"], M, D), ("w1", inp["w1"], H, D), ("w2", inp["w2"], D, H),
                                   ("dy", inp["dy"], M, D)):
        q = O.quantize_bf16(bits, fmt, hadamard=True)
        row, col = (name + "_row", name + "_col") if name in ("x", "dy") else (name + "_row", name + "t_row")
        assert_quant_equal(V[row], (q["row_payload"], q["row_scales"]), rows, cols // 32, row)
        assert_quant_equal(V[col], (q["col_payload"], q["col_scales"]), cols, rows // 32, col)

    # FC1 + bias + GELU on the chain's own X and W1
    fwd = O.gelu_fwd(_deq(V["x_row"], fmt), _deq(V["w1_row"], fmt), b1, fmt, True)
    pre_bits = _bits(V["z"])
    _close(O.bf16_to_f64(pre_bits), fwd["pre"], "pre")
    (p2, a2r, a2c), tap = with_tap(mx, M, H, lambda: mx.mx_gemm_gelu_fwd(V["x_row"], V["w1_row"], t["b1"], fmt=fmt,
                                                                           hadamard=True))
    assert torch.equal(p2, V["z"]), "pre differs between the step and the stage"
    assert torch.equal(a2r.data, V["h_row"].data) and torch.equal(a2c.data, V["h_col"].data), \
        "activation bytes differ between the step and the stage"
    assert_tap_requant_exact(V["h_row"], V["h_col"], tap, M, H, M, fmt, True, what="act")
    _close(tap.astype(np.float64), fwd["act"], "act (fp32 before the requant)")

    # FC2 + bias on the chain's own activation and W2
    y_ref = _deq(V["h_row"], fmt) @ _deq(V["w2_row"], fmt).T + b2[None, :]
    _close(bf16_cpu(out["y"]), y_ref, "y")
    db2_ref = O.colsum(O.bf16_to_f64(inp["dy"]))
    _close(out["db2"].cpu().numpy().astype(np.float64)[None, :], db2_ref[None, :], "db2")

    # FC2 dgrad + dGELU on the chain's own dY, W2^T and saved pre
    bwd = O.dgelu_bwd(_deq(V["dy_row"], fmt), _deq(V["w2t_row"], fmt), pre_bits, fmt, True)
    (d2r, d2c, _), tap = with_tap(mx, M, H, lambda: mx.mx_gemm_dgelu_bwd(V["dy_row"], V["w2t_row"], V["z"], fmt=fmt,
                                                                           hadamard=True))
    assert torch.equal(d2r.data, V["dz_row"].data) and torch.equal(d2c.data, V["dz_col"].data), \
        "dpre bytes differ between the step and the stage"
    assert_tap_requant_exact(V["dz_row"], V["dz_col"], tap, M, H, M, fmt, True, what="dpre")
    _close(tap.astype(np.float64), bwd["dpre"], "dpre (fp32 before the requant)")
    _close(out["db1"].cpu().numpy().astype(np.float64)[None, :], bwd["db1"][None, :], "db1")

    # FC1 dgrad and the weight gradients on the chain's own operands
    _close(bf16_cpu(out["dx"]), _deq(V["dz_row"], fmt) @ _deq(V["w1t_row"], fmt).T, "dx")
    _close(bf16_cpu(out["dw2"]), _deq(V["dy_col"], fmt) @ _deq(V["h_col"], fmt).T, "dw2")
    _close(bf16_cpu(out["dw1"]), _deq(V["dz_col"], fmt) @ _deq(V["x_col"], fmt).T, "dw1")


@pytest.mark.parametrize("counts", [[0, 0, 0, 0], [0, 1024, 0, 0]])
def test_swiglu_step_degenerate_routing(cuda_lib, counts):
    """No routed rows at all (every expert empty, R rows of inactive tail),
    and every routed row on one expert: the step runs clean; with no rows
    y and dX stay untouched and both weight gradients are exactly zero; with
    one expert the other experts' gradient slices are exactly zero and the
    busy expert's dW2 is held to the oracle on the step's own operands."""
    import torch
    mx = cuda_lib
    G, D, F, R = 4, 512, 256, 1152
    offsets = _offsets(counts)
    A = int(offsets[-1])
    inp = W.moe_inputs(G, D, F, R, seed=23)
    t = {k: to_dev(v) for k, v in inp.items()}
    out = {"y": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda"),
           "dx": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda"),
           "dw1": torch.full((G, 2 * F, D), float("nan"), dtype=torch.bfloat16, device="cuda"),
           "dw2": torch.full((G, D, F), float("nan"), dtype=torch.bfloat16, device="cuda")}
    offs = torch.from_numpy(offsets).cuda()
    a0 = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"], out["dw2"])
    ws = torch.zeros(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device="cuda")
    args = mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                       out["dw2"], workspace=ws)
    mx.mx_mlp_fwd_bwd(args)
    assert mx.mx_get_device_status() == "MX_OK"
    y, dx = bf16_cpu(out["y"]), bf16_cpu(out["dx"])
    assert np.isnan(y[A:]).all() and np.isnan(dx[A:]).all(), "rows past the routed segments were written"
    assert np.isfinite(y[:A]).all() and np.isfinite(dx[:A]).all()
    dw1, dw2 = bf16_cpu(out["dw1"]), bf16_cpu(out["dw2"])
    for g in range(G):
        if counts[g] == 0:
            assert (dw1[g] == 0).all() and (dw2[g] == 0).all(), "empty expert %d" % g
    if A:
        g = int(np.flatnonzero(counts)[0])
        V = mx.mlp_workspace_views(args, ws)
        E = O.E4M3
        dyc = _deq(V["dy_col"], E)[:, :A]   # [D, A]
        hc = _deq(V["h_col"], E)[:, :A]     # [F, A]
        _close(dw2[g], dyc @ hc.T, "dW2 of the busy expert")
