"""Shared test helpers: moving seeded BF16 inputs to the GPU and reading
library outputs back for comparison with the oracle."""
import numpy as np

import oracle as O


def to_dev(bits, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_cpu(t):
    """BF16 torch tensor -> float64 numpy (exact)."""
    import torch
    return O.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def mx_bytes(m):
    return m.data.cpu().numpy(), m.scale.cpu().numpy()


def assert_quant_equal(gpu_mx, ref, rows, scale_cols, what):
    """Payload and scale bytes identical (scales compared over the logical
    [rows, scale_cols] matrix and the zero padding)."""
    gp, gs = mx_bytes(gpu_mx)
    rp, rs = ref
    assert gp.shape == rp.shape, (what, gp.shape, rp.shape)
    bad = np.argwhere(gp != rp)
    assert bad.size == 0, "%s payload: %d bytes differ, first at %s (gpu %s, oracle %s)" % (
        what, len(bad), bad[0], hex(gp[tuple(bad[0])]), hex(rp[tuple(bad[0])]))
    assert gs.shape == rs.shape, (what, gs.shape, rs.shape)
    badsc = np.flatnonzero(gs != rs)
    assert badsc.size == 0, "%s scales: %d bytes differ, first at %d (gpu %s, oracle %s)" % (
        what, badsc.size, badsc[0], hex(gs[badsc[0]]), hex(rs[badsc[0]]))


def decoded(payload, scales, rows, cols, fmt=O.E4M3):
    return O.dequantize_rows(payload, scales, rows, cols, fmt)


def requant_close(gpu, ref, rows, cols, fmt=O.E4M3, max_step_frac=1e-2):
    """Fused requant from fp32 epilogue values: codes may differ from the
    oracle's only by one quantization step, where the fp32 value sits at a
    rounding boundary; returns the fraction of differing codes."""
    gp, gs = gpu
    rp, rs = ref
    gd = decoded(gp, gs, rows, cols, fmt)
    rd = decoded(rp, rs, rows, cols, fmt)
    sm = np.maximum(O.scales_to_matrix(gs, rows, cols // 32), O.scales_to_matrix(rs, rows, cols // 32))
    scale = np.repeat(2.0 ** (sm.astype(np.float64) - 127), 32, axis=1)
    step = scale * {O.E4M3: 32.0, O.E2M3: 0.5, O.E2M1: 2.0}[fmt]   # largest code spacing x scale
    diff = np.abs(gd - rd)
    assert np.all((diff <= step) | (np.isnan(gd) & np.isnan(rd))), "requant differs by more than one step"
    frac = float(np.mean(gp != rp))
    assert frac <= max_step_frac, "requant code mismatch fraction %.4f" % frac
    return frac


def assert_tap_requant_exact(gpu_row, gpu_col, tap, rows, cols, R, fmt=O.E4M3, had=False, what="tap"):
    """The fused epilogue's own fp32 values (the debug tap, [rows, cols])
    quantized by the oracle must give the epilogue's row and column bytes
    exactly.  gpu_row is [R, cols] and gpu_col [cols, R] with R >= rows; only
    the first `rows` rows (a multiple of 128) are compared."""
    x = np.asarray(tap[:rows], dtype=np.float64)
    rp, rs = O.quantize_rows(x, fmt, had)
    gp, gs = mx_bytes(gpu_row)
    assert np.array_equal(gp[:rows], rp), "%s rowwise payload differs in %d bytes" % (
        what, int((gp[:rows] != rp).sum()))
    assert np.array_equal(gs[:rs.size], rs), "%s rowwise scales differ" % what
    cp_ref, cs_ref = O.quantize_cols(x, fmt, had)
    cp, cs = mx_bytes(gpu_col)
    pb = O.payload_row_bytes(rows, fmt)
    assert np.array_equal(cp[:, :pb], cp_ref), "%s columnwise payload differs in %d bytes" % (
        what, int((cp[:, :pb] != cp_ref).sum()))
    got_s = O.scales_to_matrix(cs, cols, R // 32)[:, :rows // 32]
    assert np.array_equal(got_s, O.scales_to_matrix(cs_ref, cols, rows // 32)), "%s columnwise scales differ" % what


def with_tap(mx, rows, cols, fn):
    """Run fn with a NaN-filled fp32 debug tap [rows, cols] attached; returns
    (fn's result, the tap as float32 numpy)."""
    import torch
    tap = torch.full((rows, cols), float("nan"), dtype=torch.float32, device="cuda")
    mx.mx_debug_tap(tap)
    try:
        out = fn()
    finally:
        mx.mx_debug_tap(None)
    return out, tap.cpu().numpy()
