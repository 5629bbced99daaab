"""Grouped-GEMM parity: the CUDA GEMMs and fused epilogues against the
oracle, stage by stage, on operands quantized identically on both sides
(the quantizer's bit-exactness is asserted first)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, assert_tap_requant_exact, bf16_cpu, mx_bytes, requant_close, to_dev, with_tap

pytestmark = pytest.mark.gpu


def _quant_both(mx, bits, row=True, col=False, fmt=O.E4M3, had=False):
    """GPU and oracle rowwise (and columnwise) quantization; asserts equality."""
    x = to_dev(bits)
    r, c, _ = mx.mx_quantize(x, fmt, row, col, had)
    ref = O.quantize_bf16(bits, fmt, row, col, had)
    rows, cols = bits.shape[-2], bits.shape[-1]
    batch = bits.shape[0] if bits.ndim == 3 else 1
    if row:
        assert_quant_equal(r, (ref["row_payload"].reshape(-1, ref["row_payload"].shape[-1]),
                               ref["row_scales"].reshape(-1)), batch * rows, cols // 32, "row")
    if col:
        assert_quant_equal(c, (ref["col_payload"].reshape(-1, ref["col_payload"].shape[-1]),
                               ref["col_scales"].reshape(-1)), batch * cols, rows // 32, "col")
    return r, c, ref


def _deq(ref_key_payload, ref_key_scales, rows, cols, fmt=O.E4M3):
    return O.dequantize_rows(ref_key_payload.reshape(rows, -1), ref_key_scales.reshape(-1), rows, cols, fmt)


def _offsets(counts):
    return W.offsets_from_counts(counts)


def test_pr_ref_single_gemm(cuda_lib):
    """Single expert, X, W [256, 256] ~ N(0, 1): Y = X W^T in BF16."""
    import torch
    xb, wb = W.pr_ref(256)
    xr, _, xref = _quant_both(cuda_lib, xb)
    wr, _, wref = _quant_both(cuda_lib, wb)
    offs = torch.tensor([256], dtype=torch.int32, device="cuda")
    y = cuda_lib.mx_grouped_gemm(xr, wr, 1, offs)
    ref = _deq(xref["row_payload"], xref["row_scales"], 256, 256) @ \
        _deq(wref["row_payload"], wref["row_scales"], 256, 256).T
    got = bf16_cpu(y)
    assert O.within_tolerance(got, ref).all()
    # exact: BF16 of the exact product is what a correct fp32 accumulation rounds to, almost everywhere
    assert np.mean(got == O.bf16_out(ref)) > 0.99


@pytest.mark.parametrize("N", [512, 384])
def test_grouped_gemm_ragged(cuda_lib, N):
    """4 experts (one empty), K = 1024 (pipeline wraps), ragged inactive tail
    rows poisoned with NaN must stay untouched."""
    import torch
    G, K, R = 4, 1024, 1152
    counts = [384, 0, 256, 384]          # 1024 active rows, 128-row tail
    offsets = _offsets(counts)
    rng = np.random.default_rng(21)
    ab = W.normal_bf16(rng, (R, K))
    bb = W.normal_bf16(rng, (G, N, K), std=0.02)
    ar, _, aref = _quant_both(cuda_lib, ab)
    br, _, bref = _quant_both(cuda_lib, bb)
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(ar, br, G, torch.from_numpy(offsets).cuda(), out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    a = _deq(aref["row_payload"], aref["row_scales"], R, K)
    b = _deq(bref["row_payload"], bref["row_scales"], G * N, K).reshape(G, N, K)
    ref = O.grouped_gemm(a, b, offsets)
    got = bf16_cpu(out)
    A = int(offsets[-1])
    assert O.within_tolerance(got[:A], ref[:A]).all()
    assert np.all(np.isnan(got[A:])), "inactive tail rows were written"


@pytest.mark.parametrize("fmt", [O.E2M3, O.E2M1])
@pytest.mark.parametrize("had", [False, True])
def test_grouped_gemm_packed_formats(cuda_lib, fmt, had):
    """E2M3 / E2M1 operands (packed payload, expanded by the tensor-map
    types) with and without the 32-point rotation along K."""
    import torch
    G, K, N, R = 2, 768, 256, 512
    offsets = _offsets([256, 256])
    rng = np.random.default_rng(40 + fmt)
    ab = W.normal_bf16(rng, (R, K))
    bb = W.normal_bf16(rng, (G, N, K), std=0.02)
    ar, _, aref = _quant_both(cuda_lib, ab, fmt=fmt, had=had)
    br, _, bref = _quant_both(cuda_lib, bb, fmt=fmt, had=had)
    out = cuda_lib.mx_grouped_gemm(ar, br, G, torch.from_numpy(offsets).cuda())
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    a = _deq(aref["row_payload"], aref["row_scales"], R, K, fmt)
    b = _deq(bref["row_payload"], bref["row_scales"], G * N, K, fmt).reshape(G, N, K)
    ref = O.grouped_gemm(a, b, offsets)
    got = bf16_cpu(out)
    assert O.within_tolerance(got, ref).all()
    if had:
        # the rotation cancels in the product: compare with the unrotated one
        plain = O.grouped_gemm(O.bf16_to_f64(ab), O.bf16_to_f64(bb), offsets)
        assert O.sqnr_db(plain, got) > (20.0 if fmt == O.E2M3 else 10.0)


def test_wgrad_ragged_with_zero_token_expert(cuda_lib):
    import torch
    G, N, K, R = 4, 256, 384, 1152
    counts = [256, 0, 512, 256]
    offsets = _offsets(counts)
    A = int(offsets[-1])
    rng = np.random.default_rng(22)
    a_bits = W.normal_bf16(rng, (R, N), std=1e-3)   # e.g. dY [R, D]
    b_bits = W.normal_bf16(rng, (R, K))             # e.g. h  [R, F]
    _, ac, aref = _quant_both(cuda_lib, a_bits, row=False, col=True)
    _, bc, bref = _quant_both(cuda_lib, b_bits, row=False, col=True)
    out = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, torch.from_numpy(offsets).cuda(), out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    a_col = _deq(aref["col_payload"], aref["col_scales"], N, R)
    b_col = _deq(bref["col_payload"], bref["col_scales"], K, R)
    ref = O.wgrad(a_col, b_col, offsets)
    got = bf16_cpu(out)
    assert np.all(got[1] == 0.0), "zero-token expert must give an exactly zero slice"
    assert O.within_tolerance(got, ref).all()


@pytest.mark.parametrize("K", [384, 512])
def test_wgrad_into_fp32_main_grad_store_and_accumulate(cuda_lib, K):
    """The wgrad written into a caller's fp32 gradient buffer: the store gives
    the same accumulator the BF16 path rounds (so BF16 of it equals that
    output bit for bit) and exact zeros for an empty expert; the accumulate
    adds it with one fp32 rounding, leaves an empty expert's slice untouched,
    and onto zeros equals the store bit for bit.  K = 384 runs 128-column
    tiles, K = 512 256-column tiles."""
    import torch
    G, N, R = 4, 256, 1152
    counts = [256, 0, 512, 256]
    offsets = _offsets(counts)
    rng = np.random.default_rng(23)
    a_bits = W.normal_bf16(rng, (R, N), std=1e-3)
    b_bits = W.normal_bf16(rng, (R, K))
    _, ac, aref = _quant_both(cuda_lib, a_bits, row=False, col=True)
    _, bc, bref = _quant_both(cuda_lib, b_bits, row=False, col=True)
    offs = torch.from_numpy(offsets).cuda()
    ref = O.wgrad(_deq(aref["col_payload"], aref["col_scales"], N, R),
                  _deq(bref["col_payload"], bref["col_scales"], K, R), offsets)
    stored = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_f32(ac, bc, G, offs, stored, accumulate=False)
    bf = cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    got = stored.cpu().numpy().astype(np.float64)
    assert np.all(got[1] == 0.0)
    assert O.within_tolerance(got, ref).all()
    assert torch.equal(stored.to(torch.bfloat16), bf), "fp32 store and BF16 output disagree"
    zeros = torch.zeros((G, N, K), dtype=torch.float32, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_f32(ac, bc, G, offs, zeros, accumulate=True)
    assert torch.equal(zeros, stored), "accumulate onto zeros differs from the store"
    g0 = torch.from_numpy(rng.standard_normal((G, N, K)).astype(np.float32) * float(np.std(ref))).cuda()
    acc = g0.clone()
    cuda_lib.mx_grouped_gemm_wgrad_f32(ac, bc, G, offs, acc, accumulate=True)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    g0n = g0.cpu().numpy().astype(np.float64)
    a = acc.cpu().numpy().astype(np.float64)
    assert np.array_equal(a[1], g0n[1]), "an empty expert's slice must stay untouched"
    # one fp32 rounding of (g0 + fp32 accumulator): within the GEMM tolerance of g0 + ref
    want = g0n + ref
    err = np.abs(a - want)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * rms + 2.0 ** -23 * np.abs(want)
    assert np.all(err <= bound)
    exact = (g0 + stored).cpu()
    assert torch.equal(acc.cpu(), exact), "accumulate is not fl32(grad + stored accumulator)"


def _moe_small(seed=0, F=384):
    """Four experts (one empty), R = 1152 routed rows.  F = 384 runs the
    dSwiGLU kernel on 128-column tiles, F = 512 on 256-column ones."""
    G, D, R = 4, 1024, 1152
    counts = [384, 0, 256, 384]
    inp = W.moe_inputs(G, D, F, R, seed=seed)
    return G, D, F, R, _offsets(counts), inp


def test_swiglu_fwd_random(cuda_lib):
    import torch
    G, D, F, R, offsets, inp = _moe_small()
    A = int(offsets[-1])
    xr, _, xref = _quant_both(cuda_lib, inp["x"])
    wr, _, wref = _quant_both(cuda_lib, inp["w1"])
    z = torch.full((R, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
    z, h_row, h_col = cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, torch.from_numpy(offsets).cuda(), z=z)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    x = _deq(xref["row_payload"], xref["row_scales"], R, D)
    w = _deq(wref["row_payload"], wref["row_scales"], G * 2 * F, D).reshape(G, 2 * F, D)
    ref = O.swiglu_fwd(x, w, offsets)
    zg = bf16_cpu(z)
    assert O.within_tolerance(zg[:A], ref["z"][:A]).all()
    assert np.all(np.isnan(zg[A:])), "inactive tail of z was written"
    hp, hs = mx_bytes(h_row)
    requant_close((hp[:A], hs), ref["h_row"], A, F)
    cp, cs = mx_bytes(h_col)
    # compare the active columns of h_col [F, R] through the logical scale matrix
    got = O.dequantize_rows(cp, cs, F, R, O.E4M3)[:, :A]
    want = O.dequantize_rows(*ref["h_col"], F, A, O.E4M3)
    scale = np.repeat(2.0 ** (O.scales_to_matrix(cs, F, R // 32)[:, :A // 32].astype(np.float64) - 127), 32, axis=1)
    assert np.all(np.abs(got - want) <= scale * 32.0)
    assert np.mean(cp[:, :A] != ref["h_col"][0]) < 1e-2


def test_swiglu_fwd_exact_product_bit_exact(cuda_lib):
    """Small-integer operands make every product and partial sum exact in
    fp32 and the gate >= 64 saturates sigmoid to 1.0, so h = g*u exactly and
    the requantized bytes must match the oracle bit for bit."""
    import torch
    G, D, F, R = 2, 256, 128, 512
    rng = np.random.default_rng(31)
    x = rng.integers(1, 3, size=(R, D)).astype(np.float32)                 # 1 or 2
    w1 = np.zeros((G, 2 * F, D), dtype=np.float32)
    w1[:, :F, :64] = 1.0                                                     # gate = sum of 64 x's >= 64
    w1[:, F:, :] = rng.integers(-1, 2, size=(G, F, D)).astype(np.float32)   # up in [-512, 512]
    xb, w1b = W.to_bf16_bits(x), W.to_bf16_bits(w1)
    offsets = np.array([256, 512], dtype=np.int32)
    xr, _, xref = _quant_both(cuda_lib, xb)
    wr, _, wref = _quant_both(cuda_lib, w1b)
    z, h_row, h_col = cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, torch.from_numpy(offsets).cuda())
    xd = _deq(xref["row_payload"], xref["row_scales"], R, D)
    wd = _deq(wref["row_payload"], wref["row_scales"], G * 2 * F, D).reshape(G, 2 * F, D)
    assert np.array_equal(xd, x) and np.array_equal(wd, w1)   # exact operands
    ref = O.swiglu_fwd(xd, wd, offsets)
    assert np.array_equal(bf16_cpu(z), O.bf16_out(ref["z"]))
    assert_quant_equal(h_row, ref["h_row"], R, F // 32, "h_row")
    assert_quant_equal(h_col, ref["h_col"], F, R // 32, "h_col")


def test_dswiglu_bwd_random(cuda_lib):
    import torch
    G, D, F, R, offsets, inp = _moe_small(seed=1)
    A = int(offsets[-1])
    dyr, _, dyref = _quant_both(cuda_lib, inp["dy"])
    w2t_bits = np.ascontiguousarray(np.transpose(inp["w2"], (0, 2, 1)))   # [G, F, D]
    w2tr, _, wref = _quant_both(cuda_lib, w2t_bits)
    zb = W.normal_bf16(np.random.default_rng(5), (R, 2 * F), std=2.0)
    dz_row, dz_col = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, w2tr, to_dev(zb), G,
                                                          torch.from_numpy(offsets).cuda())
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    dy = _deq(dyref["row_payload"], dyref["row_scales"], R, D)
    w2t = _deq(wref["row_payload"], wref["row_scales"], G * F, D).reshape(G, F, D)
    ref = O.dswiglu_bwd(dy, w2t, zb, offsets)
    rp, rs = mx_bytes(dz_row)
    requant_close((rp[:A], rs), ref["dz_row"], A, 2 * F)
    cp, cs = mx_bytes(dz_col)
    got = O.dequantize_rows(cp, cs, 2 * F, R, O.E4M3)[:, :A]
    want = O.dequantize_rows(*ref["dz_col"], 2 * F, A, O.E4M3)
    scale = np.repeat(2.0 ** (O.scales_to_matrix(cs, 2 * F, R // 32)[:, :A // 32].astype(np.float64) - 127), 32,
                      axis=1)
    assert np.all(np.abs(got - want) <= scale * 32.0)
    assert np.mean(cp[:, :A] != ref["dz_col"][0]) < 1e-2


def test_dswiglu_bwd_exact_product_bit_exact(cuda_lib):
    """Saturated gates (g >= 64: sigmoid = 1 exactly) and small-integer dY,
    W2 make dg = dh*u and du = dh*g exact: bytes must match bit for bit."""
    import torch
    G, D, F, R = 2, 256, 128, 512
    rng = np.random.default_rng(32)
    dy = rng.integers(-2, 3, size=(R, D)).astype(np.float32)
    w2t = rng.integers(-1, 2, size=(G, F, D)).astype(np.float32)
    z = np.concatenate([rng.integers(64, 128, size=(R, F)), rng.integers(-8, 9, size=(R, F))], axis=1)
    dyb, w2tb, zb = W.to_bf16_bits(dy), W.to_bf16_bits(w2t), W.to_bf16_bits(z.astype(np.float32))
    offsets = np.array([128, 512], dtype=np.int32)
    dyr, _, dyref = _quant_both(cuda_lib, dyb)
    w2tr, _, wref = _quant_both(cuda_lib, w2tb)
    dz_row, dz_col = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, w2tr, to_dev(zb), G,
                                                          torch.from_numpy(offsets).cuda())
    dyd = _deq(dyref["row_payload"], dyref["row_scales"], R, D)
    w2td = _deq(wref["row_payload"], wref["row_scales"], G * F, D).reshape(G, F, D)
    assert np.array_equal(dyd, dy) and np.array_equal(w2td, w2t)
    ref = O.dswiglu_bwd(dyd, w2td, zb, offsets)
    assert_quant_equal(dz_row, ref["dz_row"], R, 2 * F // 32, "dz_row")
    assert_quant_equal(dz_col, ref["dz_col"], 2 * F, R // 32, "dz_col")


def test_swiglu_fwd_tap_requant_bit_exact(cuda_lib):
    """Random inputs: the epilogue's own fp32 h (debug tap), quantized by the
    oracle, gives h_row and h_col bit for bit; the tap is the oracle's h
    within the GEMM tolerance and the inactive tail rows are never written."""
    import torch
    G, D, F, R, offsets, inp = _moe_small(seed=3)
    A = int(offsets[-1])
    xr, _, xref = _quant_both(cuda_lib, inp["x"])
    wr, _, wref = _quant_both(cuda_lib, inp["w1"])
    offs = torch.from_numpy(offsets).cuda()
    (z, h_row, h_col), tap = with_tap(cuda_lib, R, F, lambda: cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, offs))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert_tap_requant_exact(h_row, h_col, tap, A, F, R, what="h")
    assert np.all(np.isnan(tap[A:])), "tail rows of the tap were written"
    x = _deq(xref["row_payload"], xref["row_scales"], R, D)
    w = _deq(wref["row_payload"], wref["row_scales"], G * 2 * F, D).reshape(G, 2 * F, D)
    ref = O.swiglu_fwd(x, w, offsets)
    assert O.within_tolerance(tap[:A].astype(np.float64), ref["h"]).all()


@pytest.mark.parametrize("F", [256, 384, 512])
def test_dswiglu_bwd_tap_requant_bit_exact_and_gate_up_swap_fails(cuda_lib, F):
    """Random inputs: the epilogue's fp32 dz = [dg | du] (debug tap) quantized
    by the oracle gives dz_row and dz_col bit for bit, and matches the
    oracle's dz within tolerance.  Negative control: the oracle with gate and
    up swapped in z must not match."""
    import torch
    G, D, F, R, offsets, inp = _moe_small(seed=4, F=F)
    A = int(offsets[-1])
    dyr, _, dyref = _quant_both(cuda_lib, inp["dy"])
    w2t_bits = np.ascontiguousarray(np.transpose(inp["w2"], (0, 2, 1)))
    w2tr, _, wref = _quant_both(cuda_lib, w2t_bits)
    zb = W.normal_bf16(np.random.default_rng(6), (R, 2 * F), std=2.0)
    offs = torch.from_numpy(offsets).cuda()
    (dz_row, dz_col), tap = with_tap(cuda_lib, R, 2 * F,
                                     lambda: cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, w2tr, to_dev(zb), G, offs))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert_tap_requant_exact(dz_row, dz_col, tap, A, 2 * F, R, what="dz")
    assert np.all(np.isnan(tap[A:]))
    dy = _deq(dyref["row_payload"], dyref["row_scales"], R, D)
    w2t = _deq(wref["row_payload"], wref["row_scales"], G * F, D).reshape(G, F, D)
    ref = O.dswiglu_bwd(dy, w2t, zb, offsets)
    got = tap[:A].astype(np.float64)
    assert O.within_tolerance(got, ref["dz"]).all()
    swapped = np.ascontiguousarray(np.concatenate([zb[:, F:], zb[:, :F]], axis=1))
    bad = O.dswiglu_bwd(dy, w2t, swapped, offsets)
    assert np.mean(O.within_tolerance(got, bad["dz"])) < 0.5, "gate/up swap went unnoticed"


def _same_active(a, b, A, cols, R, what):
    """Two requant outputs agree on the active rows (row orientation [R, cols])
    or active columns (column orientation [cols, R]); rows and columns past
    the last segment are never written."""
    ar, ac = a
    br, bc = b
    assert np.array_equal(ar.data.cpu().numpy()[:A], br.data.cpu().numpy()[:A]), what
    sr = O.scales_to_matrix(ar.scale.cpu().numpy(), R, cols // 32)[:A]
    assert np.array_equal(sr, O.scales_to_matrix(br.scale.cpu().numpy(), R, cols // 32)[:A]), what
    assert np.array_equal(ac.data.cpu().numpy()[:, :A], bc.data.cpu().numpy()[:, :A]), what
    sc = O.scales_to_matrix(ac.scale.cpu().numpy(), cols, R // 32)[:, :A // 32]
    assert np.array_equal(sc, O.scales_to_matrix(bc.scale.cpu().numpy(), cols, R // 32)[:, :A // 32]), what


@pytest.mark.parametrize("F", [384, 512])
def test_swiglu_with_routing_probabilities(cuda_lib, F):
    """The fused activation with routing probabilities, forward and backward:
    probs = 1 reproduces the plain kernels' bytes exactly; random probs give
    requant bytes bit-exact given the epilogue's own fp32 values (debug tap),
    those values within tolerance of the oracle, and dprobs within tolerance
    of the oracle's sum_f dh * swiglu(g, u), the same on a second run."""
    import torch
    G, D, F, R, offsets, inp = _moe_small(seed=7, F=F)
    A = int(offsets[-1])
    offs = torch.from_numpy(offsets).cuda()
    xr, _, xref = _quant_both(cuda_lib, inp["x"])
    wr, _, wref = _quant_both(cuda_lib, inp["w1"])
    probs_np = np.random.default_rng(8).uniform(0.05, 1.0, R).astype(np.float32)
    probs = torch.from_numpy(probs_np).cuda()
    ones = torch.ones(R, dtype=torch.float32, device="cuda")
    z0, h0r, h0c = cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, offs)
    z1, h1r, h1c = cuda_lib.mx_grouped_gemm_swiglu_probs_fwd(xr, wr, G, offs, ones)
    assert torch.equal(z0[:A], z1[:A])
    _same_active((h0r, h0c), (h1r, h1c), A, F, R, "h with probs = 1")
    (z, h_row, h_col), tap = with_tap(cuda_lib, R, F,
                                      lambda: cuda_lib.mx_grouped_gemm_swiglu_probs_fwd(xr, wr, G, offs, probs))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert_tap_requant_exact(h_row, h_col, tap, A, F, R, what="h*p")
    x = _deq(xref["row_payload"], xref["row_scales"], R, D)
    w = _deq(wref["row_payload"], wref["row_scales"], G * 2 * F, D).reshape(G, 2 * F, D)
    ref = O.swiglu_fwd(x, w, offsets, probs=probs_np.astype(np.float64))
    assert O.within_tolerance(tap[:A].astype(np.float64), ref["h"]).all()

    dyr, _, dyref = _quant_both(cuda_lib, inp["dy"])
    w2t_bits = np.ascontiguousarray(np.transpose(inp["w2"], (0, 2, 1)))
    w2tr, _, w2ref = _quant_both(cuda_lib, w2t_bits)
    d0r, d0c = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, w2tr, z, G, offs)
    d1r, d1c, _ = cuda_lib.mx_grouped_gemm_dswiglu_probs_bwd(dyr, w2tr, z, ones, G, offs)
    _same_active((d0r, d0c), (d1r, d1c), A, 2 * F, R, "dz with probs = 1")
    dprobs0 = torch.full((R,), float("nan"), dtype=torch.float32, device="cuda")
    (dz_row, dz_col, dprobs), tap2 = with_tap(
        cuda_lib, R, 2 * F,
        lambda: cuda_lib.mx_grouped_gemm_dswiglu_probs_bwd(dyr, w2tr, z, probs, G, offs, dprobs=dprobs0))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert_tap_requant_exact(dz_row, dz_col, tap2, A, 2 * F, R, what="dz with probs")
    dy = _deq(dyref["row_payload"], dyref["row_scales"], R, D)
    w2t = _deq(w2ref["row_payload"], w2ref["row_scales"], G * F, D).reshape(G, F, D)
    zb = z.view(torch.int16).cpu().numpy().view(np.uint16)
    bref = O.dswiglu_bwd(dy, w2t, zb, offsets, probs=probs_np.astype(np.float64))
    assert O.within_tolerance(tap2[:A].astype(np.float64), bref["dz"]).all()
    got = dprobs.cpu().numpy().astype(np.float64)
    assert np.all(np.isnan(got[A:])), "rows past the segments were written"
    assert O.within_tolerance(got[None, :A], bref["dprobs"][None, :]).all()
    again = cuda_lib.mx_grouped_gemm_dswiglu_probs_bwd(dyr, w2tr, z, probs, G, offs)[2]
    assert torch.equal(again[:A], dprobs[:A]), "dprobs is not deterministic"


@pytest.mark.parametrize("F", [384, 512])
def test_mlp_step_against_oracle_chain(cuda_lib, F):
    """The whole SwiGLU step through mx_mlp_fwd_bwd against the oracle's
    chain (F = 512 runs dSwiGLU on 256-column tiles)."""
    import torch
    G, D, F, R, offsets, inp = _moe_small(seed=2, F=F)
    A = int(offsets[-1])
    t = {k: to_dev(v) for k, v in inp.items()}
    dev = "cuda"
    out = {"y": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device=dev),
           "dx": torch.full((R, D), float("nan"), dtype=torch.bfloat16, device=dev),
           "dw1": torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device=dev),
           "dw2": torch.empty((G, D, F), dtype=torch.bfloat16, device=dev)}
    offs = torch.from_numpy(offsets).cuda()
    args = cuda_lib.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                             out["dw2"])
    ws = torch.empty(cuda_lib.mx_mlp_workspace_bytes(args), dtype=torch.uint8, device=dev)
    args = cuda_lib.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                             out["dw2"], workspace=ws)
    cuda_lib.mx_mlp_fwd_bwd(args)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = O.mlp_fwd_bwd_swiglu(inp["x"], inp["w1"], inp["w2"], inp["dy"], offsets)
    unq = O.mlp_fwd_bwd_swiglu_unquantized(inp["x"], inp["w1"], inp["w2"], inp["dy"], offsets)
    got = {k: bf16_cpu(v) for k, v in out.items()}
    assert np.all(np.isnan(got["y"][A:])) and np.all(np.isnan(got["dx"][A:]))
    assert np.all(got["dw1"][1] == 0) and np.all(got["dw2"][1] == 0)
    for k in ("y", "dx", "dw1", "dw2"):
        g = got[k][:A] if k in ("y", "dx") else got[k]
        s_orc = O.sqnr_db(ref[k + "_f64"], g)
        s_unq = O.sqnr_db(unq[k], g)
        assert s_orc > 35.0, (k, s_orc)
        # the torchao PR #5 page's MXFP8 chain band (y 23.7 dB) minus 6 dB
        assert s_unq > 23.7 - 6.0, (k, s_unq)
    # z, read back from the step's workspace: its band (28.5 dB) minus 6 dB
    zg = bf16_cpu(cuda_lib.mlp_workspace_views(args, ws)["z"])[:A]
    assert O.sqnr_db(unq["z"], zg) > 28.5 - 6.0
    # run-to-run bitwise determinism
    first = {k: v.clone() for k, v in out.items()}
    cuda_lib.mx_mlp_fwd_bwd(args)
    for k in out:
        assert torch.equal(torch.nan_to_num(first[k]), torch.nan_to_num(out[k])), k


def test_bounded_wait_reports_timeout(cuda_lib):
    cuda_lib.mx_selftest_bounded_wait(50_000_000)   # 50 ms, nothing will arrive
    assert cuda_lib.mx_get_device_status() == "MX_ERR_DEVICE_TIMEOUT"
    assert cuda_lib.mx_get_device_status() == "MX_OK"


def test_r_zero_and_g_zero(cuda_lib):
    import torch
    a = cuda_lib.MX(0, 256)
    b = cuda_lib.MX(256, 256)
    offs = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(a, b, 1, offs, out=out, ld_out=256)
    with pytest.raises(cuda_lib.MXError) as e:
        cuda_lib.mx_grouped_gemm(a, b, 0, offs, out=out, ld_out=256)
    assert e.value.name == "MX_ERR_INVALID_ARG"


@pytest.mark.parametrize("fmt,N", [(O.E4M3, 384), (O.E4M3, 512), (O.E2M1, 256)])
def test_grouped_gemm_per_expert_bias(cuda_lib, fmt, N):
    """Each segment gets its own expert's bias row in the fp32 accumulator
    (4 experts, one empty, NaN-poisoned inactive tail untouched); E2M1 runs
    the kind::mxf4 path.  Small-integer operands and biases make the sums
    exact, so the BF16 output is compared bit for bit."""
    import torch
    G, K, R = 4, 512, 1152
    offsets = _offsets([384, 0, 256, 384])
    rng = np.random.default_rng(120 + N + fmt)
    a = rng.integers(-2, 3, size=(R, K)).astype(np.float32)
    b = rng.integers(-2, 3, size=(G, N, K)).astype(np.float32)
    bias = rng.integers(-64, 65, size=(G, N)).astype(np.float32)
    ar, _, aref = _quant_both(cuda_lib, W.to_bf16_bits(a), fmt=fmt)
    br, _, bref = _quant_both(cuda_lib, W.to_bf16_bits(b), fmt=fmt)
    assert np.array_equal(_deq(aref["row_payload"], aref["row_scales"], R, K, fmt), a)
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bias_dev = torch.from_numpy(W.to_bf16_bits(bias).view(np.int16)).cuda().view(torch.bfloat16)
    cuda_lib.mx_grouped_gemm_bias(ar, br, G, torch.from_numpy(offsets).cuda(), bias_dev, out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = O.grouped_gemm_bias(a.astype(np.float64), b.astype(np.float64), bias.astype(np.float64), offsets)
    A = int(offsets[-1])
    got = bf16_cpu(out)
    assert np.array_equal(got[:A], O.bf16_out(ref[:A]))
    assert np.all(np.isnan(got[A:]))


@pytest.mark.parametrize("fmt,K", [(O.E4M3, 384), (O.E4M3, 512), (O.E2M1, 384)])
def test_wgrad_k_split_exact_and_deterministic(cuda_lib, fmt, K):
    """An expert with 20480 tokens (160 chunks of 128) has its K range split
    into parts reduced by the last part to arrive.  Small-integer operands
    make every partial sum exact, so BF16 out, the fp32 store and the fp32
    accumulate must equal the oracle bit for bit (K = 384: 128-column
    tiles, K = 512: 256-column tiles; E2M1 runs kind::mxf4)."""
    import torch
    G, N = 4, 256
    counts = [20480, 0, 1024, 512]
    offsets = _offsets(counts)
    R = int(offsets[-1])
    rng = np.random.default_rng(130 + K + fmt)
    a = rng.integers(-2, 3, size=(R, N)).astype(np.float32)
    b = rng.integers(-2, 3, size=(R, K)).astype(np.float32)
    _, ac, aref = _quant_both(cuda_lib, W.to_bf16_bits(a), row=False, col=True, fmt=fmt)
    _, bc, bref = _quant_both(cuda_lib, W.to_bf16_bits(b), row=False, col=True, fmt=fmt)
    assert cuda_lib.mx_grouped_gemm_wgrad_workspace_bytes(N, K, R, G) > 0
    offs = torch.from_numpy(offsets).cuda()
    ref = O.wgrad(a.T.astype(np.float64), b.T.astype(np.float64), offsets)
    out = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_ws(ac, bc, G, offs, out=out)
    st = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_f32_ws(ac, bc, G, offs, st, accumulate=False)
    g0 = torch.from_numpy(rng.integers(-8, 9, size=(G, N, K)).astype(np.float32)).cuda()
    acc = g0.clone()
    cuda_lib.mx_grouped_gemm_wgrad_f32_ws(ac, bc, G, offs, acc, accumulate=True)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert np.array_equal(bf16_cpu(out), O.bf16_out(ref))
    assert np.array_equal(st.cpu().numpy().astype(np.float64), ref)
    assert np.array_equal(acc.cpu().numpy().astype(np.float64), g0.cpu().numpy().astype(np.float64) + ref)


def test_wgrad_k_split_random_is_deterministic_and_close_to_unsplit(cuda_lib):
    """Random operands: the split wgrad gives the same bits on every run,
    agrees with the oracle within the GEMM tolerance, and with the unsplit
    call to fp32 summation order (BF16 outputs within one BF16 step)."""
    import torch
    G, N, K = 4, 256, 512
    counts = [20480, 0, 1024, 512]
    offsets = _offsets(counts)
    R = int(offsets[-1])
    rng = np.random.default_rng(140)
    _, ac, aref = _quant_both(cuda_lib, W.normal_bf16(rng, (R, N), std=1e-3), row=False, col=True)
    _, bc, bref = _quant_both(cuda_lib, W.normal_bf16(rng, (R, K)), row=False, col=True)
    offs = torch.from_numpy(offsets).cuda()
    runs = [cuda_lib.mx_grouped_gemm_wgrad_ws(ac, bc, G, offs) for _ in range(3)]
    plain = cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert all(torch.equal(runs[0], r) for r in runs[1:]), "split wgrad is not deterministic"
    ref = O.wgrad(_deq(aref["col_payload"], aref["col_scales"], N, R), _deq(bref["col_payload"], bref["col_scales"], K, R),
                  offsets)
    got = bf16_cpu(runs[0])
    assert np.all(got[1] == 0.0)
    assert O.within_tolerance(got, ref).all()
    p = bf16_cpu(plain)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    assert np.all(np.abs(got - p) <= 2.0 ** -7 * np.abs(p) + 2.0 ** -14 * rms)


def test_wgrad_claimed_tiles_equal_dealt_tiles(cuda_lib):
    """With a workspace the wgrad's CTAs claim tiles from a counter instead
    of taking a fixed share.  With no expert large enough to be split
    (64 experts of at most 1024 rows, several empty: over a thousand tiles,
    several per CTA) every tile is still computed once by one CTA, so the
    result equals the call without a workspace bit for bit, on every run."""
    import torch
    G, N, K = 64, 256, 512
    rng = np.random.default_rng(160)
    counts = [int(c) for c in rng.integers(0, 9, size=G) * 128]
    counts[3] = counts[17] = 0
    offsets = _offsets(counts)
    R = int(offsets[-1])
    _, ac, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (R, N), std=1e-3), row=False, col=True)
    _, bc, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (R, K)), row=False, col=True)
    offs = torch.from_numpy(offsets).cuda()
    plain = cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, offs)
    runs = []
    for _ in range(3):
        out = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        runs.append(cuda_lib.mx_grouped_gemm_wgrad_ws(ac, bc, G, offs, out=out))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    for r in runs:
        assert torch.equal(r, plain), "claimed tiles differ from dealt tiles"
    assert (plain[3] == 0).all() and (plain[17] == 0).all()


def test_wgrad_k_split_writes_nothing_outside_its_output(cuda_lib):
    """The split wgrad launches headroom tiles for the parts; tiles past the
    last expert must stay inactive: poisoned guard slices around the output
    (in one allocation) stay untouched, and an empty expert's slice is zero."""
    import torch
    G, N, K = 4, 256, 384
    offsets = _offsets([20480, 0, 1024, 512])
    R = int(offsets[-1])
    rng = np.random.default_rng(150)
    _, ac, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (R, N), std=1e-3), row=False, col=True)
    _, bc, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (R, K)), row=False, col=True)
    buf = torch.full((G + 4, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[2:2 + G]
    cuda_lib.mx_grouped_gemm_wgrad_ws(ac, bc, G, torch.from_numpy(offsets).cuda(), out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert torch.isnan(buf[:2]).all() and torch.isnan(buf[2 + G:]).all()
    assert (out[1] == 0).all() and not torch.isnan(out).any()


def test_malformed_offsets_reported_on_device_and_opt_in_host_check(cuda_lib, monkeypatch):
    """Offsets that are not multiples of 128: by default the call launches,
    the kernels skip the malformed segments (their rows stay untouched) and
    mx_get_device_status reports MX_ERR_OFFSETS once; with
    MX_VALIDATE_OFFSETS=1 the host reads the offsets first and returns
    MX_ERR_OFFSETS without launching."""
    import torch
    G, K, N, R = 2, 256, 256, 512
    rng = np.random.default_rng(160)
    ar, _, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (R, K)))
    br, _, _ = _quant_both(cuda_lib, W.normal_bf16(rng, (G, N, K), std=0.02))
    bad = torch.tensor([100, 256], dtype=torch.int32, device="cuda")
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(ar, br, G, bad, out=out)
    assert cuda_lib.mx_get_device_status() == "MX_ERR_OFFSETS"
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert torch.isnan(out[:256]).all(), "rows of malformed segments were written"
    monkeypatch.setenv("MX_VALIDATE_OFFSETS", "1")
    with pytest.raises(cuda_lib.MXError) as e:
        cuda_lib.mx_grouped_gemm(ar, br, G, bad, out=out)
    assert e.value.name == "MX_ERR_OFFSETS"
    dec = torch.tensor([256, 128], dtype=torch.int32, device="cuda")
    with pytest.raises(cuda_lib.MXError) as e:
        cuda_lib.mx_grouped_gemm(ar, br, G, dec, out=out)
    assert e.value.name == "MX_ERR_OFFSETS" and "decreases" in str(e.value)
    good = torch.tensor([256, 512], dtype=torch.int32, device="cuda")
    cuda_lib.mx_grouped_gemm(ar, br, G, good, out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M3, O.E2M1])
def test_one_hot_probe_tensor_core_reads_our_element_order(cuda_lib, fmt):
    """Row i of A is one-hot at K position i (i < 256: every position of
    eight 32-element blocks, both nibbles / all four 6-bit slots of each
    packed group), B holds distinct small integers; then Y[i, n] must be
    B[n, i] exactly.  A packing-order or scale-slot mismatch between our
    payload layout and the tensor core's reading moves values to other K
    positions and fails here position by position (E2M1 runs kind::mxf4)."""
    import torch
    K, N = 256, 256
    a = np.zeros((256, K), dtype=np.float32)
    a[np.arange(256), np.arange(256)] = 1.0
    n_idx, k_idx = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    b = (((n_idx * 5 + k_idx * 3) % 7) - 3).astype(np.float32)          # -3..3, exact in every format
    ar, _, aref = _quant_both(cuda_lib, W.to_bf16_bits(a), fmt=fmt)
    br, _, bref = _quant_both(cuda_lib, W.to_bf16_bits(b), fmt=fmt)
    assert np.array_equal(_deq(aref["row_payload"], aref["row_scales"], 256, K, fmt), a)
    assert np.array_equal(_deq(bref["row_payload"], bref["row_scales"], N, K, fmt), b)
    y = cuda_lib.mx_gemm_bias(ar, br, None)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    got = bf16_cpu(y)
    bad = np.argwhere(got != b.T)
    assert bad.size == 0, "first wrong (row=K position, n): %s" % bad[:4].tolist()
