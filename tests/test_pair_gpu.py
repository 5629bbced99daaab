"""The CTA-pair grouped GEMM (mx_grouped_gemm_2sm) and the 256-row routing
it needs.

Each product is the single-SM kernel's (the same K order of block-scaled
MMAs into fp32), so the pair's outputs must equal mx_grouped_gemm's bit for
bit, besides matching the oracle within the benchmark spec's tolerance."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_quant_equal, bf16_cpu, to_dev

pytestmark = pytest.mark.gpu


def _quant(mx, bits, fmt=O.E4M3, had=False):
    x = to_dev(bits)
    r, _, _ = mx.mx_quantize(x, fmt, True, False, had)
    ref = O.quantize_bf16(bits, fmt, True, False, had)
    rows, cols = bits.shape[-2], bits.shape[-1]
    batch = bits.shape[0] if bits.ndim == 3 else 1
    assert_quant_equal(r, (ref["row_payload"].reshape(-1, ref["row_payload"].shape[-1]),
                           ref["row_scales"].reshape(-1)), batch * rows, cols // 32, "row")
    return r, ref


def _deq(ref, rows, cols, fmt=O.E4M3):
    return O.dequantize_rows(ref["row_payload"].reshape(rows, -1), ref["row_scales"].reshape(-1), rows, cols, fmt)


@pytest.mark.parametrize("N,K,counts", [(512, 1024, [512, 0, 256, 768]), (256, 768, [512, 0, 256, 768]),
                                         (512, 768, [384, 128, 0, 640])])
def test_pair_gemm_equals_single_sm_and_oracle(cuda_lib, N, K, counts):
    """4 experts with a 256-row inactive tail poisoned with NaN (K = 1024
    wraps the six-stage ring); segments of 256-row multiples, or of odd
    128-row block counts (384, 128, 640: each expert's last 256-row tile
    computes an upper half past its segment, which must not be stored)."""
    import torch
    mx = cuda_lib
    G, R = 4, 1792
    offsets = W.offsets_from_counts(counts)
    A = int(offsets[-1])
    rng = np.random.default_rng(51 + N)
    ab = W.normal_bf16(rng, (R, K))
    bb = W.normal_bf16(rng, (G, N, K), std=0.02)
    ar, aref = _quant(mx, ab)
    br, bref = _quant(mx, bb)
    offs = torch.from_numpy(offsets).cuda()
    pair = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.mx_grouped_gemm_2sm(ar, br, G, offs, out=pair)
    single = mx.mx_grouped_gemm(ar, br, G, offs)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    assert torch.equal(pair[:A], single[:A]), "pair and single-SM products differ"
    got = bf16_cpu(pair)
    ref = O.grouped_gemm(_deq(aref, R, K), _deq(bref, G * N, K).reshape(G, N, K), offsets)
    assert O.within_tolerance(got[:A], ref[:A]).all()
    assert np.all(np.isnan(got[A:])), "inactive tail rows were written"


def test_pair_gemm_exact_products(cuda_lib):
    """Small-integer operands times powers of two: every partial sum is
    exact in fp32, so the BF16 output equals the oracle's exact product
    rounded once."""
    import torch
    mx = cuda_lib
    G, N, K, R = 2, 256, 512, 512
    offsets = W.offsets_from_counts([256, 256])
    rng = np.random.default_rng(7)
    a = rng.integers(-3, 4, size=(R, K)).astype(np.float32) * np.float32(2.0 ** -2)
    b = rng.integers(-3, 4, size=(G, N, K)).astype(np.float32) * np.float32(2.0 ** 1)
    ab, bb = W.to_bf16_bits(a), W.to_bf16_bits(b)
    ar, aref = _quant(mx, ab)
    br, bref = _quant(mx, bb)
    out = mx.mx_grouped_gemm_2sm(ar, br, G, torch.from_numpy(offsets).cuda())
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    ref = O.grouped_gemm(_deq(aref, R, K), _deq(bref, G * N, K).reshape(G, N, K), offsets)
    assert np.array_equal(bf16_cpu(out), O.bf16_out(ref))


@pytest.mark.parametrize("had", [False, True])
def test_pair_gemm_dense_e2m3(cuda_lib, had):
    """One segment of all rows (no offsets), E2M3 operands with and without
    the rotation along K."""
    import torch
    mx = cuda_lib
    R, N, K = 512, 512, 768
    rng = np.random.default_rng(9)
    ab = W.normal_bf16(rng, (R, K))
    bb = W.normal_bf16(rng, (N, K), std=0.02)
    ar, aref = _quant(mx, ab, O.E2M3, had)
    br, bref = _quant(mx, bb, O.E2M3, had)
    pair = mx.mx_grouped_gemm_2sm(ar, br, 1, None)
    single = mx.mx_grouped_gemm(ar, br, 1, None)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    assert torch.equal(pair, single)
    ref = _deq(aref, R, K, O.E2M3) @ _deq(bref, N, K, O.E2M3).T
    assert O.within_tolerance(bf16_cpu(pair), ref).all()


def test_pair_gemm_reports_malformed_segments(cuda_lib):
    """A segment that is not a multiple of 128 rows (and every segment after
    it that starts off the grid) is skipped on the device, its rows left
    untouched, and the call's status reads MX_ERR_OFFSETS; the well-formed
    expert before it is computed."""
    import torch
    mx = cuda_lib
    G, N, K, R = 3, 256, 256, 768
    offsets = np.array([256, 456, 640], dtype=np.int32)   # expert 1 ends, expert 2 starts, off the grid
    rng = np.random.default_rng(3)
    ar, _ = _quant(mx, W.normal_bf16(rng, (R, K)))
    br, _ = _quant(mx, W.normal_bf16(rng, (G, N, K), std=0.02))
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.mx_grouped_gemm_2sm(ar, br, G, torch.from_numpy(offsets).cuda(), out=out)
    assert mx.mx_get_device_status() == "MX_ERR_OFFSETS"
    assert mx.mx_get_device_status() == "MX_OK"
    good = W.offsets_from_counts([256, 0, 0])
    single = mx.mx_grouped_gemm(ar, br, G, torch.from_numpy(good).cuda())
    torch.cuda.synchronize()
    assert torch.equal(out[:256], single[:256])
    assert bool(torch.isnan(out[256:].float()).all())


def test_route_index_pads_to_256(cuda_lib):
    """The routing index with 256-row segments equals the oracle's exactly."""
    import torch
    mx = cuda_lib
    T, k, G = 4096, 8, 64
    rng = np.random.default_rng(17)
    pop = 1.0 / np.arange(1, G + 1) ** 1.1
    topk = np.stack([rng.choice(G, size=k, replace=False, p=pop / pop.sum()) for _ in range(T)]).astype(np.int32)
    offs, src, row_of = mx.mx_moe_route_index(torch.from_numpy(topk).cuda(), G, pad=256)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    o_offs, o_src, o_row = O.moe_route_index(topk, G, pad=256)
    assert np.array_equal(offs.cpu().numpy(), o_offs)
    R = int(o_offs[-1])
    assert np.array_equal(src.cpu().numpy()[:R], o_src)
    assert np.all(src.cpu().numpy()[R:] == -1)
    assert np.array_equal(row_of.cpu().numpy(), o_row)
    assert np.all(o_offs % 256 == 0)


def test_pair_gemm_e2m1_exact_products(cuda_lib):
    """Packed E2M1 operands on .kind::mxf4: integers in [-3, 3] times powers
    of two quantize exactly to E2M1 and every partial sum is exact in fp32,
    so the BF16 output equals the oracle's exact product rounded once, and
    the single-SM kernel's bit for bit."""
    import torch
    mx = cuda_lib
    G, N, K, R = 2, 256, 768, 512
    offsets = W.offsets_from_counts([256, 256])
    rng = np.random.default_rng(11)
    a = rng.integers(-3, 4, size=(R, K)).astype(np.float32) * np.float32(2.0 ** -3)
    b = rng.integers(-3, 4, size=(G, N, K)).astype(np.float32) * np.float32(2.0 ** 2)
    ar, aref = _quant(mx, W.to_bf16_bits(a), O.E2M1)
    br, bref = _quant(mx, W.to_bf16_bits(b), O.E2M1)
    offs = torch.from_numpy(offsets).cuda()
    pair = mx.mx_grouped_gemm_2sm(ar, br, G, offs)
    single = mx.mx_grouped_gemm(ar, br, G, offs)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    ref = O.grouped_gemm(_deq(aref, R, K, O.E2M1), _deq(bref, G * N, K, O.E2M1).reshape(G, N, K), offsets)
    assert np.array_equal(bf16_cpu(pair), O.bf16_out(ref))
    assert torch.equal(pair, single)


@pytest.mark.parametrize("K,counts", [(640, [512, 0, 256]), (1024, [512, 0, 256]), (640, [128, 0, 640])])
def test_pair_gemm_e2m1_ragged(cuda_lib, K, counts):
    """E2M1 on random operands with a NaN-poisoned inactive tail; K = 640
    ends on half a stage (five 128-K chunks), K = 1024 wraps the five-stage
    ring; segments of 256-row multiples or of odd 128-row block counts.
    Bit-identical to the single-SM .kind::mxf4 kernel and within tolerance
    of the oracle."""
    import torch
    mx = cuda_lib
    G, N, R = 3, 512, 1024
    offsets = W.offsets_from_counts(counts)
    A = int(offsets[-1])
    rng = np.random.default_rng(K)
    ar, aref = _quant(mx, W.normal_bf16(rng, (R, K)), O.E2M1)
    br, bref = _quant(mx, W.normal_bf16(rng, (G, N, K), std=0.02), O.E2M1)
    offs = torch.from_numpy(offsets).cuda()
    pair = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.mx_grouped_gemm_2sm(ar, br, G, offs, out=pair)
    single = mx.mx_grouped_gemm(ar, br, G, offs)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    assert torch.equal(pair[:A], single[:A]), "pair and single-SM products differ"
    got = bf16_cpu(pair)
    ref = O.grouped_gemm(_deq(aref, R, K, O.E2M1), _deq(bref, G * N, K, O.E2M1).reshape(G, N, K), offsets)
    assert O.within_tolerance(got[:A], ref[:A]).all()
    assert np.all(np.isnan(got[A:])), "inactive tail rows were written"


@pytest.mark.parametrize("fmt,had,counts", [(O.E4M3, False, [384, 0, 256]), (O.E2M3, True, [256, 128, 256])])
def test_pair_gemm_bias_equals_single_sm(cuda_lib, fmt, had, counts):
    """The bias epilogue on CTA pairs (each expert's BF16 bias row added to
    the fp32 accumulator before the one rounding) equals the single-SM bias
    epilogue bit for bit, rows past the segments untouched."""
    import torch
    mx = cuda_lib
    G, N, K, R = 3, 512, 768, 1024
    offsets = W.offsets_from_counts(counts)
    A = int(offsets[-1])
    rng = np.random.default_rng(29)
    ar, _ = _quant(mx, W.normal_bf16(rng, (R, K)), fmt, had)
    br, _ = _quant(mx, W.normal_bf16(rng, (G, N, K), std=0.02), fmt, had)
    bias = to_dev(W.normal_bf16(rng, (G, N), std=0.5))
    offs = torch.from_numpy(offsets).cuda()
    pair = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.mx_grouped_gemm_bias_2sm(ar, br, G, offs, bias, out=pair)
    single = mx.mx_grouped_gemm_bias(ar, br, G, offs, bias)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    assert torch.equal(pair[:A], single[:A])
    assert bool(torch.isnan(pair[A:].float()).all())
