"""Quantizer parity: the CUDA quantizer's payload and scale bytes must equal
the oracle's, bit for bit, on seeded inputs with special values."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, to_dev

pytestmark = pytest.mark.gpu

FMTS = [O.E4M3, O.E2M3, O.E2M1]


def _run(mx, bits, fmt, row=True, col=True, had=False):
    x = to_dev(bits)
    return mx.mx_quantize(x, fmt, row, col, had)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("rows,cols", [(256, 256), (96, 160), (288, 224), (32, 32), (640, 384)])
def test_quantize_bytes_match_oracle(cuda_lib, fmt, had, rows, cols):
    bits = W.quantizer_input(rows, cols, seed=rows * 7 + cols, special_frac=0.01)
    xr, xc, _ = _run(cuda_lib, bits, fmt, True, True, had)
    ref = O.quantize_bf16(bits, fmt, True, True, had)
    assert_quant_equal(xr, (ref["row_payload"], ref["row_scales"]), rows, cols // 32, "row")
    assert_quant_equal(xc, (ref["col_payload"], ref["col_scales"]), cols, rows // 32, "col")


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_pattern(cuda_lib, fmt):
    """All 65536 BF16 patterns, laid out so each lands in many blocks."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    rng = np.random.default_rng(3)
    for perm_seed in range(2):
        b = bits.reshape(-1)[rng.permutation(1 << 16)].reshape(256, 256) if perm_seed else bits
        xr, xc, _ = _run(cuda_lib, b, fmt)
        ref = O.quantize_bf16(b, fmt)
        assert_quant_equal(xr, (ref["row_payload"], ref["row_scales"]), 256, 8, "row")
        assert_quant_equal(xc, (ref["col_payload"], ref["col_scales"]), 256, 8, "col")


def test_negative_controls_flipped_byte_and_floor_scales(cuda_lib):
    """The byte gate must catch one flipped scale byte and one flipped payload
    byte planted in the oracle's reference, and the GPU's scales must differ
    from FLOOR scales (derived from the oracle's) on most blocks while
    equalling RCEIL exactly."""
    rows, cols = 256, 256
    bits = W.quantizer_input(rows, cols, seed=9, special_frac=0.0)
    xr, _, _ = _run(cuda_lib, bits, O.E4M3, True, False)
    ref = O.quantize_bf16(bits, O.E4M3, True, False)
    good = (ref["row_payload"], ref["row_scales"])
    assert_quant_equal(xr, good, rows, cols // 32, "row")
    bad_scale = ref["row_scales"].copy()
    bad_scale[O.blocked_offset(5, 3, cols // 32)] ^= 1
    with pytest.raises(AssertionError):
        assert_quant_equal(xr, (ref["row_payload"], bad_scale), rows, cols // 32, "row")
    bad_payload = ref["row_payload"].copy()
    bad_payload[17, 33] ^= 0x01
    with pytest.raises(AssertionError):
        assert_quant_equal(xr, (bad_payload, ref["row_scales"]), rows, cols // 32, "row")
    x = O.bf16_to_f64(bits)
    amax = np.max(np.abs(x.reshape(rows, cols // 32, 32)), axis=2)
    emax = O.fmt_max(O.E4M3)
    rceil = np.vectorize(lambda a: O.scale_byte(a, O.E4M3))(amax)
    exact_pow = amax == emax * 2.0 ** (rceil.astype(np.float64) - 127)
    floor = rceil - (~exact_pow).astype(rceil.dtype)
    got = O.scales_to_matrix(xr.scale.cpu().numpy(), rows, cols // 32)
    assert np.array_equal(got, rceil)
    assert np.mean(got != floor) > 0.9


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1])
def test_rowwise_only_and_colwise_only(cuda_lib, fmt):
    bits = W.quantizer_input(160, 256, seed=5, special_frac=0.01)
    xr, xc, _ = _run(cuda_lib, bits, fmt, True, False)
    assert xc is None
    ref = O.quantize_bf16(bits, fmt, True, True)
    assert_quant_equal(xr, (ref["row_payload"], ref["row_scales"]), 160, 8, "row")
    xr, xc, _ = _run(cuda_lib, bits, fmt, False, True)
    assert xr is None
    assert_quant_equal(xc, (ref["col_payload"], ref["col_scales"]), 256, 5, "col")


def test_strided_input(cuda_lib):
    import torch
    bits = W.quantizer_input(128, 512, seed=9, special_frac=0.0)
    full = to_dev(bits)
    x = full[:, 64:320]          # ld = 512, cols = 256
    xr, xc, _ = cuda_lib.mx_quantize(x, O.E4M3, True, True)
    ref = O.quantize_bf16(np.ascontiguousarray(bits[:, 64:320]), O.E4M3)
    assert_quant_equal(xr, (ref["row_payload"], ref["row_scales"]), 128, 8, "row")
    assert_quant_equal(xc, (ref["col_payload"], ref["col_scales"]), 256, 4, "col")
    assert torch.equal(full, to_dev(bits))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M3, O.E2M1])
def test_batched_weights(cuda_lib, fmt):
    """[G, N, K] weights: rowwise of the stack and per-expert columnwise."""
    G, N, K = 3, 256, 384
    bits = W.normal_bf16(np.random.default_rng(4), (G, N, K), std=0.02)
    xr, xc, _ = _run(cuda_lib, bits, fmt)
    rp, rs = O.quantize_experts_rows(bits, fmt)
    cp, cs = O.quantize_experts_cols(bits, fmt)
    assert_quant_equal(xr, (rp, rs), G * N, K // 32, "row")
    assert_quant_equal(xc, (cp, cs), G * K, N // 32, "col")


@pytest.mark.parametrize("rows,cols", [(1024, 256), (96, 160)])
def test_colsum(cuda_lib, rows, cols):
    import torch
    bits = W.normal_bf16(np.random.default_rng(6), (rows, cols), std=1e-3)
    x = to_dev(bits)
    xr, xc, cs = cuda_lib.mx_quantize(x, O.E2M3, True, True, True, True)
    ref = O.colsum(O.bf16_to_f64(bits))
    got = cs.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * np.sqrt(np.mean(ref ** 2)))
    # determinism: the fixed-order reduction is bitwise repeatable
    _, _, cs2 = cuda_lib.mx_quantize(x, O.E2M3, True, True, True, True)
    assert torch.equal(cs, cs2)


def test_rows_zero_is_a_no_op(cuda_lib):
    import torch
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    out_row = cuda_lib.MX(0, 64)
    out_col = cuda_lib.MX(64, 0)
    cuda_lib.mx_quantize(x, O.E4M3, True, True, out_row=out_row, out_col=out_col)


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1])
def test_quantizer_workload_full_size(cuda_lib, fmt):
    """The standalone quantizer workload at full size: 8192 x 7168 BF16,
    heavy-tailed rows spanning 2^+-20, 0.1 % specials; MXFP8 and MXFP4,
    both orientations, every byte compared."""
    bits = W.quantizer_input(**W.QUANT_SHAPE)
    xr, xc, _ = _run(cuda_lib, bits, fmt)
    ref = O.quantize_bf16(bits, fmt)
    assert_quant_equal(xr, (ref["row_payload"], ref["row_scales"]), 8192, 7168 // 32, "row")
    assert_quant_equal(xc, (ref["col_payload"], ref["col_scales"]), 7168, 8192 // 32, "col")


def _oracle_sr(bits, fmt, seed, had):
    """Oracle stochastic-rounding quantization of BF16 [rows, cols] or
    [batch, rows, cols]: rowwise over [batch*rows, cols], columnwise over the
    stacked per-batch transposes [batch*cols, rows]."""
    x = O.bf16_to_f64(bits)
    if x.ndim == 2:
        x = x[None]
    B, rows, cols = x.shape
    row = O.quantize_rows_sr(x.reshape(B * rows, cols), fmt, seed, 0, had)
    col = O.quantize_rows_sr(np.concatenate([x[b].T for b in range(B)], axis=0), fmt, seed, 1, had)
    return row, col


@pytest.mark.parametrize("fmt", [O.E2M3, O.E2M1])
@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("shape", [(256, 256), (96, 160), (2, 128, 256)])
def test_stochastic_rounding_bytes_match_oracle(cuda_lib, fmt, had, shape):
    """mx_quantize_sr against the oracle's stochastic rounding (Philox bits per
    element of each output grid), bit for bit, specials included; a 64-bit
    seed with high bits set exercises both key words."""
    if len(shape) == 3:
        bits = np.stack([W.quantizer_input(shape[1], shape[2], seed=70 + b, special_frac=0.01) for b in range(shape[0])])
    else:
        bits = W.quantizer_input(shape[0], shape[1], seed=71, special_frac=0.01)
    seed = 0x9E3779B97F4A7C15
    r, c = cuda_lib.mx_quantize_sr(to_dev(bits), fmt, seed, True, shape[-2] % 32 == 0, had)
    ref_row, ref_col = _oracle_sr(bits, fmt, seed, had)
    B = shape[0] if len(shape) == 3 else 1
    rows, cols = shape[-2], shape[-1]
    assert_quant_equal(r, ref_row, B * rows, cols // 32, "sr row")
    if rows % 32 == 0:
        assert_quant_equal(c, ref_col, B * cols, rows // 32, "sr col")


def test_stochastic_rounding_seed_dependence(cuda_lib):
    """Same seed, same bytes; another seed, other bytes (scales unchanged)."""
    import torch
    bits = W.quantizer_input(256, 256, seed=72, special_frac=0.0)
    x = to_dev(bits)
    a = cuda_lib.mx_quantize_sr(x, O.E2M1, 1)[0]
    b = cuda_lib.mx_quantize_sr(x, O.E2M1, 1)[0]
    c = cuda_lib.mx_quantize_sr(x, O.E2M1, 2)[0]
    assert torch.equal(a.data, b.data) and torch.equal(a.scale, b.scale)
    assert torch.equal(a.scale, c.scale)
    assert float((a.data != c.data).float().mean()) > 0.2


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [O.E2M1, O.E2M3])
def test_stochastic_rounding_full_size_workload(cuda_lib, fmt):
    """Stochastic rounding on the full 8192 x 7168 workload (heavy-tailed
    rows, 0.1 % specials), both orientations, every byte against the
    oracle's Philox-driven rounding."""
    bits = W.quantizer_input(**W.QUANT_SHAPE)
    r, c = cuda_lib.mx_quantize_sr(to_dev(bits), fmt, 0x5EED, True, True)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    row, col = _oracle_sr(bits, fmt, 0x5EED, False)
    rows, cols = bits.shape
    assert_quant_equal(r, row, rows, cols // 32, "row")
    assert_quant_equal(c, col, cols, rows // 32, "col")
