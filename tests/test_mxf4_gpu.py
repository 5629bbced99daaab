"""MXFP4 (E2M1) GEMMs on the packed-operand tensor-core path (.kind::mxf4)
against the oracle: grouped, dense with bias, ragged-K wgrad into BF16 and
into an fp32 main-grad buffer.  A pipeline stage covers 256 K-elements, so
K ranges with an odd number of 128-element chunks end on a half stage; the
shapes below exercise both, and both 128- and 256-column tiles."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, bf16_cpu, to_dev

pytestmark = pytest.mark.gpu

E2M1 = O.E2M1


def _q(mx, bits, row=True, col=False):
    """GPU and oracle E2M1 quantization (asserted equal); dequantized oracle
    operands in float64."""
    r, c, _ = mx.mx_quantize(to_dev(bits), E2M1, row, col)
    ref = O.quantize_bf16(bits, E2M1, row, col)
    rows, cols = bits.shape[-2], bits.shape[-1]
    batch = bits.shape[0] if bits.ndim == 3 else 1
    out = {}
    if row:
        pay, sc = ref["row_payload"].reshape(batch * rows, -1), ref["row_scales"].reshape(-1)
        assert_quant_equal(r, (pay, sc), batch * rows, cols // 32, "row")
        out["row"] = O.dequantize_rows(pay, sc, batch * rows, cols, E2M1)
    if col:
        pay, sc = ref["col_payload"].reshape(batch * cols, -1), ref["col_scales"].reshape(-1)
        assert_quant_equal(c, (pay, sc), batch * cols, rows // 32, "col")
        out["col"] = O.dequantize_rows(pay, sc, batch * cols, rows, E2M1)
    return r, c, out


def _small_ints(rng, shape, lo=-3, hi=3):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


@pytest.mark.parametrize("K,N", [(640, 384), (640, 512), (128, 256), (1024, 256)])
def test_mxf4_grouped_gemm_ragged(cuda_lib, K, N):
    """Random operands, 4 experts (one empty), inactive tail rows poisoned
    with NaN stay untouched; K = 640 and 128 end on a half stage."""
    import torch
    G, R = 4, 1152
    offsets = W.offsets_from_counts([384, 0, 256, 384])
    rng = np.random.default_rng(60 + K + N)
    ar, _, a = _q(cuda_lib, W.normal_bf16(rng, (R, K)))
    br, _, b = _q(cuda_lib, W.normal_bf16(rng, (G, N, K), std=0.02))
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(ar, br, G, torch.from_numpy(offsets).cuda(), out=out)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = O.grouped_gemm(a["row"], b["row"].reshape(G, N, K), offsets)
    got = bf16_cpu(out)
    A = int(offsets[-1])
    assert O.within_tolerance(got[:A], ref[:A]).all()
    assert np.all(np.isnan(got[A:])), "inactive tail rows were written"


@pytest.mark.parametrize("K", [1152, 1280])
def test_mxf4_exact_products_bit_exact(cuda_lib, K):
    """Small-integer operands quantize exactly to E2M1 and every product and
    partial sum is exact in fp32, so the BF16 output must equal the oracle's
    rounding of the exact result bit for bit (K = 1152: nine chunks, a half
    last stage)."""
    import torch
    G, N, R = 2, 256, 512
    offsets = np.array([256, 512], dtype=np.int32)
    rng = np.random.default_rng(K)
    x, w = _small_ints(rng, (R, K)), _small_ints(rng, (G, N, K))
    ar, _, a = _q(cuda_lib, W.to_bf16_bits(x))
    br, _, b = _q(cuda_lib, W.to_bf16_bits(w))
    assert np.array_equal(a["row"], x) and np.array_equal(b["row"].reshape(G, N, K), w)
    out = cuda_lib.mx_grouped_gemm(ar, br, G, torch.from_numpy(offsets).cuda())
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = O.grouped_gemm(x.astype(np.float64), w.astype(np.float64), offsets)
    assert np.array_equal(bf16_cpu(out), O.bf16_out(ref))


def test_mxf4_dense_gemm_bias(cuda_lib):
    """Dense E2M1 GEMM with a BF16 bias added to the fp32 accumulator."""
    M, N, K = 256, 384, 640
    rng = np.random.default_rng(66)
    ar, _, a = _q(cuda_lib, W.normal_bf16(rng, (M, K)))
    br, _, b = _q(cuda_lib, W.normal_bf16(rng, (N, K), std=0.02))
    bias = W.normal_bf16(rng, (N,), std=0.02)
    out = cuda_lib.mx_gemm_bias(ar, br, to_dev(bias))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = a["row"] @ b["row"].T + O.bf16_to_f64(bias)[None, :]
    assert O.within_tolerance(bf16_cpu(out), ref).all()


@pytest.mark.parametrize("N,K", [(256, 384), (256, 512)])
def test_mxf4_wgrad_bf16_and_fp32(cuda_lib, N, K):
    """Ragged-K wgrad on E2M1 columnwise operands: expert token counts 128,
    0, 384, 256 (odd and even chunk counts, an empty expert); BF16 out and
    the fp32 store / accumulate into a main-grad buffer, exact-product
    operands so every output is compared bit for bit."""
    import torch
    G, R = 4, 896
    counts = [128, 0, 384, 256]
    offsets = W.offsets_from_counts(counts)
    rng = np.random.default_rng(70 + K)
    a_bits = W.to_bf16_bits(_small_ints(rng, (R, N), -2, 2))
    b_bits = W.to_bf16_bits(_small_ints(rng, (R, K), -2, 2))
    _, ac, a = _q(cuda_lib, a_bits, row=False, col=True)
    _, bc, b = _q(cuda_lib, b_bits, row=False, col=True)
    offs = torch.from_numpy(offsets).cuda()
    ref = O.wgrad(a["col"], b["col"], offsets)
    assert np.array_equal(a["col"], W.bf16_bits_to_f32(a_bits).T)   # exact operands
    bf = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, offs, out=bf)
    stored = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_f32(ac, bc, G, offs, stored, accumulate=False)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert np.array_equal(bf16_cpu(bf), O.bf16_out(ref))
    assert np.array_equal(stored.cpu().numpy().astype(np.float64), ref)
    g0 = torch.from_numpy(rng.integers(-8, 9, size=(G, N, K)).astype(np.float32)).cuda()
    acc = g0.clone()
    cuda_lib.mx_grouped_gemm_wgrad_f32(ac, bc, G, offs, acc, accumulate=True)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert np.array_equal(acc.cpu().numpy().astype(np.float64), g0.cpu().numpy().astype(np.float64) + ref)


def test_mxf4_wgrad_random(cuda_lib):
    """Random E2M1 wgrad operands, Zipf-like ragged counts, within the
    GEMM tolerance."""
    import torch
    G, N, K, R = 4, 256, 384, 1152
    counts = [256, 0, 512, 256]
    offsets = W.offsets_from_counts(counts)
    rng = np.random.default_rng(77)
    _, ac, a = _q(cuda_lib, W.normal_bf16(rng, (R, N), std=1e-3), row=False, col=True)
    _, bc, b = _q(cuda_lib, W.normal_bf16(rng, (R, K)), row=False, col=True)
    out = cuda_lib.mx_grouped_gemm_wgrad(ac, bc, G, torch.from_numpy(offsets).cuda())
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    ref = O.wgrad(a["col"], b["col"], offsets)
    got = bf16_cpu(out)
    assert np.all(got[1] == 0.0)
    assert O.within_tolerance(got, ref).all()
