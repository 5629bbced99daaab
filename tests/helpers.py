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


def decode_lut(fmt):
    """float64 value of every unpacked element code of fmt (NaN codes give NaN)."""
    n = {O.E4M3: 256, O.E2M3: 64, O.E2M1: 16}[fmt]
    return np.array([O.decode(c, fmt) for c in range(n)])


def mx_row_scales(m, rows):
    """Scale bytes [len(rows), cols/32] of the given rows of an MX tensor
    (read from its blocked layout)."""
    import torch
    off = O.blocked_index(m.rows, m.cols // 32, rows)
    return m.scale[torch.from_numpy(off.reshape(-1)).to(m.scale.device)].cpu().numpy().reshape(off.shape)


def mx_rows_f64(m, rows, lut):
    """Dequantized rows of an E4M3 MX tensor (one payload byte per element)."""
    import torch
    idx = torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(m.data.device)
    codes = m.data[idx].cpu().numpy()
    s = mx_row_scales(m, rows).astype(np.float64)
    return lut[codes] * np.repeat(2.0 ** (s - 127.0), 32, axis=1)


def assert_tap_requant_exact_sampled(gpu_row, gpu_col, tap, rows, fmt=O.E4M3, had=False, what="tap"):
    """Sampled form of assert_tap_requant_exact for full-size outputs: the
    rowwise payload and scale bytes of `rows`, and the columnwise payload and
    scale bytes of every 32-row block holding one of them, equal the
    oracle's quantization of the epilogue's own fp32 values (the tap,
    a torch tensor [R, C] on the GPU)."""
    import torch
    rows = np.asarray(sorted(rows), dtype=np.int64)
    R, C = tap.shape
    idx = torch.from_numpy(rows).to(tap.device)
    t = tap[idx].cpu().numpy().astype(np.float64)
    rp, rs = O.quantize_rows(t, fmt, had)
    assert np.array_equal(gpu_row.data[idx].cpu().numpy(), rp), "%s rowwise payload differs" % what
    assert np.array_equal(mx_row_scales(gpu_row, rows), O.scales_to_matrix(rs, len(rows), C // 32)), \
        "%s rowwise scales differ" % what
    pb = O.payload_row_bytes(32, fmt)
    col_scales = mx_row_scales(gpu_col, np.arange(C))                    # [C, R/32]
    for b in np.unique(rows // 32):
        blk = tap[32 * b:32 * b + 32].cpu().numpy().astype(np.float64)  # [32, C]
        cp, cs = O.quantize_rows(np.ascontiguousarray(blk.T), fmt, had)  # [C, one block]
        got = gpu_col.data[:, b * pb:(b + 1) * pb].cpu().numpy()
        assert np.array_equal(got, cp), "%s columnwise payload of rows %d..%d differs" % (what, 32 * b, 32 * b + 31)
        assert np.array_equal(col_scales[:, b], O.scales_to_matrix(cs, C, 1)[:, 0]), \
            "%s columnwise scales of rows %d..%d differ" % (what, 32 * b, 32 * b + 31)
