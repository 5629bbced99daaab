"""Expert counts at and past the CTA-pair kernels' limit.

G = 1024 is the most experts the CTA-pair kernels' row-tile table holds and
the most the weight gradient ranks by size; G = 1100 runs past both: the
CTA-pair GEMM rejects it, the fused SwiGLU forward takes one SM per tile,
and the weight gradient deals its tiles in expert order with no ranking and
no K-split.  Most experts are empty and the others hold 128 to 512 rows, so
every kind of segment boundary occurs many times.  Operands are quantized by
both sides (bytes asserted equal) and the outputs held to the oracle on the
oracle's own dequantized operands."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, assert_tap_requant_exact, bf16_cpu, to_dev, with_tap

pytestmark = pytest.mark.gpu

ACTIVE = 160  # experts with rows


def _routing(G, seed):
    rng = np.random.default_rng(seed)
    counts = np.zeros(G, dtype=np.int64)
    counts[rng.choice(G, ACTIVE, replace=False)] = 128 * rng.integers(1, 5, size=ACTIVE)
    offsets = W.offsets_from_counts(counts)
    return counts, offsets, int(offsets[-1]) + 128   # a 128-row inactive tail


def _quant_rows(mx, bits):
    """GPU rowwise quantization of BF16 bits [R, C] or [B, R, C], asserted
    equal to the oracle's; returns (GPU tensor, oracle dequantized float64)."""
    r, _, _ = mx.mx_quantize(to_dev(bits), O.E4M3, True, False)
    ref = O.quantize_bf16(bits, O.E4M3, True, False)
    rows, cols = bits.shape[-2], bits.shape[-1]
    batch = bits.shape[0] if bits.ndim == 3 else 1
    p, s = ref["row_payload"].reshape(batch * rows, -1), ref["row_scales"].reshape(-1)
    assert_quant_equal(r, (p, s), batch * rows, cols // 32, "row")
    deq = O.dequantize_rows(p, s, batch * rows, cols, O.E4M3)
    return r, deq.reshape(bits.shape)


def _quant_cols(mx, bits):
    """GPU columnwise quantization of BF16 bits [R, C] (stored [C, R]),
    asserted equal to the oracle's; returns (GPU tensor, dequantized [C, R])."""
    _, c, _ = mx.mx_quantize(to_dev(bits), O.E4M3, False, True)
    ref = O.quantize_bf16(bits, O.E4M3, False, True)
    rows, cols = bits.shape
    assert_quant_equal(c, (ref["col_payload"], ref["col_scales"]), cols, rows // 32, "col")
    return c, O.dequantize_rows(ref["col_payload"], ref["col_scales"], cols, rows, O.E4M3)


@pytest.mark.parametrize("G", [1024, 1100])
def test_many_experts_grouped_gemm(cuda_lib, G):
    """y = A B[g]^T over G experts: within tolerance of the oracle, the
    inactive tail untouched; at G = 1024 the CTA-pair kernel's output equals
    the single-SM kernel's byte for byte, at G = 1100 the pair kernel refuses
    the call."""
    import torch
    counts, offsets, R = _routing(G, seed=G)
    N, K = 256, 128
    rng = np.random.default_rng(G + 1)
    ab = W.normal_bf16(rng, (R, K))
    bb = W.normal_bf16(rng, (G, N, K), std=0.02)
    ar, ad = _quant_rows(cuda_lib, ab)
    br, bd = _quant_rows(cuda_lib, bb)
    offs = torch.from_numpy(offsets).cuda()
    y = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(ar, br, G, offs, out=y)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    A = int(offsets[-1])
    got = bf16_cpu(y)
    assert O.within_tolerance(got[:A], O.grouped_gemm(ad, bd, offsets)[:A]).all()
    assert np.isnan(got[A:]).all(), "inactive tail was written"
    y2 = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if G <= 1024:
        cuda_lib.mx_grouped_gemm_2sm(ar, br, G, offs, out=y2)
        assert cuda_lib.mx_get_device_status() == "MX_OK"
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    else:
        with pytest.raises(cuda_lib.MXError, match="1024"):
            cuda_lib.mx_grouped_gemm_2sm(ar, br, G, offs, out=y2)


@pytest.mark.parametrize("G", [1024, 1100])
def test_many_experts_swiglu_fwd(cuda_lib, monkeypatch, G):
    """FC1 + SwiGLU over G experts: z within tolerance of the oracle, the
    requantized h bytes equal to the oracle's quantization of the epilogue's
    fp32 values (debug tap), and the default path (CTA pairs up to 1024
    experts, one SM per tile past it) byte-equal to one SM per tile."""
    import torch
    counts, offsets, R = _routing(G, seed=G + 2)
    D, F = 128, 128
    rng = np.random.default_rng(G + 3)
    xb = W.normal_bf16(rng, (R, D))
    wb = W.normal_bf16(rng, (G, 2 * F, D), std=0.02)
    xr, xd = _quant_rows(cuda_lib, xb)
    wr, wd = _quant_rows(cuda_lib, wb)
    offs = torch.from_numpy(offsets).cuda()
    A = int(offsets[-1])

    def run():
        h_row, h_col = cuda_lib.MX(R, F), cuda_lib.MX(F, R)
        for m in (h_row, h_col):   # the inactive tail is never written: a fixed fill on both runs
            m.data.fill_(0x5A)
            m.scale.fill_(0x5A)
        z = torch.full((R, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
        cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, offs, h_row, h_col, z)
        assert cuda_lib.mx_get_device_status() == "MX_OK"
        return z, h_row, h_col

    (z, h_row, h_col), tap = with_tap(cuda_lib, R, F, run)
    ref = O.swiglu_fwd(xd, wd, offsets)
    zg = bf16_cpu(z)
    assert O.within_tolerance(zg[:A], ref["z"][:A]).all()
    assert np.isnan(zg[A:]).all(), "inactive tail of z was written"
    assert O.within_tolerance(tap[:A], ref["h"]).all()
    assert_tap_requant_exact(h_row, h_col, tap, A, F, R, what="h")
    monkeypatch.setenv("MX_FUSED_PAIRS", "0")
    z1, h1r, h1c = run()
    for a, b in ((z, z1), (h_row.data, h1r.data), (h_row.scale, h1r.scale), (h_col.data, h1c.data),
                 (h_col.scale, h1c.scale)):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("G", [1024, 1100])
def test_many_experts_wgrad(cuda_lib, G):
    """dW[g] = A[g]^T B[g] over G experts, with the workspace (tiles claimed
    largest expert first at G = 1024; dealt in expert order past it): within
    tolerance of the oracle, every empty expert's slice exactly zero."""
    import torch
    counts, offsets, R = _routing(G, seed=G + 4)
    N, K = 256, 128
    rng = np.random.default_rng(G + 5)
    ab = W.normal_bf16(rng, (R, N), std=1e-3)
    bb = W.normal_bf16(rng, (R, K))
    ac, ad = _quant_cols(cuda_lib, ab)
    bc, bd = _quant_cols(cuda_lib, bb)
    offs = torch.from_numpy(offsets).cuda()
    dw = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_ws(ac, bc, G, offs, out=dw)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    got = bf16_cpu(dw)
    ref = O.wgrad(ad, bd, offsets)
    active = np.flatnonzero(counts)
    assert O.within_tolerance(got[active], ref[active]).all()
    assert (got[np.flatnonzero(counts == 0)] == 0).all(), "an empty expert's slice is not zero"


@pytest.mark.parametrize("G", [1024, 1100])
def test_many_experts_dswiglu_bwd(cuda_lib, G):
    """FC2 dgrad + dSwiGLU over G experts (one SM per tile, 128-column tiles
    at F = 128): the epilogue's fp32 dz (debug tap) within tolerance of the
    oracle's dSwiGLU of the exact dh and the saved z, and both requantized
    orientations equal to the oracle's quantization of those fp32 values."""
    import torch
    counts, offsets, R = _routing(G, seed=G + 6)
    D, F = 128, 128
    rng = np.random.default_rng(G + 7)
    dyb = W.normal_bf16(rng, (R, D), std=1e-3)
    w2tb = W.normal_bf16(rng, (G, F, D), std=0.02)
    zb = W.normal_bf16(rng, (R, 2 * F), std=2.0)
    dyr, dyd = _quant_rows(cuda_lib, dyb)
    w2tr, w2td = _quant_rows(cuda_lib, w2tb)
    offs = torch.from_numpy(offsets).cuda()
    A = int(offsets[-1])

    def run():
        dz_row, dz_col = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, w2tr, to_dev(zb), G, offs)
        assert cuda_lib.mx_get_device_status() == "MX_OK"
        return dz_row, dz_col

    (dz_row, dz_col), tap = with_tap(cuda_lib, R, 2 * F, run)
    ref = O.dswiglu_bwd(dyd, w2td, zb, offsets)
    assert O.within_tolerance(tap[:A], ref["dz"]).all()
    assert_tap_requant_exact(dz_row, dz_col, tap, A, 2 * F, R, what="dz")
