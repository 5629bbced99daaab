"""Full-size parity of the dense MXFP6 + Hadamard tanh-GELU stages (M=16384,
D=3072, H=12288, the benchmark's launch configuration) and of the dense
MXFP4 GEMM line (16384 x 12288 x 3072), on sampled outputs.

Sampling: two 32-row blocks x two 32-column blocks from different tiles.
Rowwise blocks span 32 columns and columnwise blocks 32 rows of one column,
so the oracle quantizes only the sampled rows / columns of each operand and
gets exactly the bytes the full quantization would give there.  Each stage
gets its own seeded BF16 inputs; no oracle input comes from the CUDA path."""
import numpy as np
import pytest

import oracle as O
from helpers import bf16_cpu, requant_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

M, D, H = 16384, 3072, 12288
E2M3 = O.E2M3
ROWS = np.r_[np.arange(4096, 4128), np.arange(12256, 12288)]     # 32-row blocks 128 and 383
COLS = np.r_[np.arange(224, 256), np.arange(9600, 9632)]         # 32-column blocks 7 and 300


def _rand_bf16(shape, std, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16)


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _idx(a):
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.int64)).cuda()


def _deq_rows(x64, fmt=E2M3, had=True):
    p, s = O.quantize_rows(x64, fmt, had)
    return O.dequantize_rows(p, s, x64.shape[0], x64.shape[1], fmt)


def _sub_row(mx_t, rows, cols, fmt=E2M3):
    """GPU rowwise tensor [R, C] -> (payload [n, 32-col blocks], blocked
    scales) of the sampled rows and 32-column blocks."""
    bb = {O.E4M3: 32, O.E2M3: 24, O.E2M1: 16}[fmt]
    blocks = np.unique(np.asarray(cols) // 32)
    pay = mx_t.data[_idx(rows)].cpu().numpy()
    pay = np.concatenate([pay[:, b * bb:(b + 1) * bb] for b in blocks], axis=1)
    sm = O.scales_to_matrix(mx_t.scale.cpu().numpy(), mx_t.rows, mx_t.cols // 32)[np.ix_(rows, blocks)]
    blocked = np.zeros(O.scale_bytes(len(rows), len(blocks)), dtype=np.uint8)
    blocked[O.blocked_index(len(rows), len(blocks))] = sm
    return pay, blocked


def _tapped(cuda_lib, fn):
    """Run fn with a NaN-filled fp32 debug tap [M, H] attached; returns
    (fn's result, the tap on the GPU)."""
    import torch
    tap = torch.full((M, H), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap)
    try:
        out = fn()
    finally:
        cuda_lib.mx_debug_tap(None)
    return out, tap


def _assert_tap_exact_blocks(tap, gpu_row, gpu_col, what):
    """The epilogue's own fp32 values on the sampled blocks (the tap, before
    the rotation), quantized by the oracle with the Hadamard rotation, give
    the sampled rowwise and columnwise payload and scale bytes exactly (the
    samples are whole 32-row and 32-column blocks)."""
    t = tap[_idx(ROWS)][:, _idx(COLS)].cpu().numpy().astype(np.float64)
    rp, rs = O.quantize_rows(t, E2M3, True)
    gp, gs = _sub_row(gpu_row, ROWS, COLS)
    assert np.array_equal(gp, rp), "%s rowwise payload differs in %d bytes" % (what, int((gp != rp).sum()))
    assert np.array_equal(gs, rs), "%s rowwise scales differ" % what
    cp, cs = O.quantize_rows(np.ascontiguousarray(t.T), E2M3, True)
    gp, gs = _sub_row(gpu_col, COLS, ROWS)
    assert np.array_equal(gp, cp), "%s columnwise payload differs in %d bytes" % (what, int((gp != cp).sum()))
    assert np.array_equal(gs, cs), "%s columnwise scales differ" % what


def test_dense_fc1_gelu_full_size_sampled_blocks(cuda_lib):
    """pre = x W1^T + b1 (BF16) within tolerance; the epilogue's fp32 act =
    gelu(pre) (debug tap) within tolerance of the oracle, and act packed
    rowwise and columnwise byte-equal to the oracle's quantization of those
    fp32 values (rotation included), on 64 x 64 samples; the packed bytes
    also within one quantization step of the oracle's own act."""
    x = _rand_bf16((M, D), 1.0, 71)
    w1 = _rand_bf16((H, D), 0.02, 72)
    b1 = _rand_bf16((H,), 0.02, 73)
    xr, _, _ = cuda_lib.mx_quantize(x, E2M3, True, False, True)
    wr, _, _ = cuda_lib.mx_quantize(w1, E2M3, True, False, True)
    (pre, act_row, act_col), tap = _tapped(cuda_lib, lambda: cuda_lib.mx_gemm_gelu_fwd(xr, wr, b1))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    xq = _deq_rows(O.bf16_to_f64(_bits(x[_idx(ROWS)])))
    wq = _deq_rows(O.bf16_to_f64(_bits(w1[_idx(COLS)])))
    ref = O.gelu_fwd(xq, wq, O.bf16_to_f64(_bits(b1))[COLS], E2M3, True)
    got = bf16_cpu(pre[_idx(ROWS)][:, _idx(COLS)])
    assert O.within_tolerance(got, ref["pre"]).all()
    t = tap[_idx(ROWS)][:, _idx(COLS)].cpu().numpy().astype(np.float64)
    assert O.within_tolerance(t, ref["act"]).all()
    _assert_tap_exact_blocks(tap, act_row, act_col, "act")
    requant_close(_sub_row(act_row, ROWS, COLS), ref["act_row"], len(ROWS), len(COLS), E2M3)
    requant_close(_sub_row(act_col, COLS, ROWS), ref["act_col"], len(COLS), len(ROWS), E2M3)


def test_dense_dgelu_full_size_sampled_blocks(cuda_lib):
    """dpre = (dY W2) * gelu'(pre) from the BF16 save: the epilogue's fp32
    dpre (debug tap) within tolerance of the oracle and packed both ways
    byte-equal to the oracle's quantization of it, on 64 x 64 samples (W2's
    columnwise quantization gives the W2^T operand)."""
    dy = _rand_bf16((M, D), 1e-3, 81)
    w2 = _rand_bf16((D, H), 0.02, 82)
    pre = _rand_bf16((M, H), 1.5, 83)
    dyr, _, _ = cuda_lib.mx_quantize(dy, E2M3, True, False, True)
    _, w2t, _ = cuda_lib.mx_quantize(w2, E2M3, False, True, True)
    (dpre_row, dpre_col, _), tap = _tapped(cuda_lib, lambda: cuda_lib.mx_gemm_dgelu_bwd(dyr, w2t, pre))
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    dyq = _deq_rows(O.bf16_to_f64(_bits(dy[_idx(ROWS)])))
    w2tq = _deq_rows(O.bf16_to_f64(_bits(w2[:, _idx(COLS)])).T.copy())
    pre_s = _bits(pre[_idx(ROWS)][:, _idx(COLS)])
    ref = O.dgelu_bwd(dyq, w2tq, pre_s, E2M3, True)
    t = tap[_idx(ROWS)][:, _idx(COLS)].cpu().numpy().astype(np.float64)
    assert O.within_tolerance(t, ref["dpre"]).all()
    _assert_tap_exact_blocks(tap, dpre_row, dpre_col, "dpre")
    requant_close(_sub_row(dpre_row, ROWS, COLS), ref["dpre_row"], len(ROWS), len(COLS), E2M3)
    requant_close(_sub_row(dpre_col, COLS, ROWS), ref["dpre_col"], len(COLS), len(ROWS), E2M3)


def test_dense_wgrad_full_size_sampled_entries(cuda_lib):
    """dW1 = dpre^T x over all 16384 rows, both operands columnwise E2M3 with
    the rotation along M, on an 8 x 8 sample of [H, D]."""
    dpre = _rand_bf16((M, H), 1e-3, 91)
    x = _rand_bf16((M, D), 1.0, 92)
    _, dpc, _ = cuda_lib.mx_quantize(dpre, E2M3, False, True, True)
    _, xc, _ = cuda_lib.mx_quantize(x, E2M3, False, True, True)
    dw1 = cuda_lib.mx_grouped_gemm_wgrad(dpc, xc, 1, None)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rng = np.random.default_rng(9)
    hs, ds = np.sort(rng.choice(H, 8, replace=False)), np.sort(rng.choice(D, 8, replace=False))
    a = _deq_rows(O.bf16_to_f64(_bits(dpre[:, _idx(hs)])).T.copy())    # [8, M]
    b = _deq_rows(O.bf16_to_f64(_bits(x[:, _idx(ds)])).T.copy())       # [8, M]
    got = bf16_cpu(dw1[0][_idx(hs)][:, _idx(ds)])
    assert O.within_tolerance(got, a @ b.T).all()


def test_mxfp4_gemm_full_size_sampled_blocks(cuda_lib):
    """The dense MXFP4 GEMM of the benchmark (16384 x 12288 x 3072, E2M1 on
    tcgen05 kind::mxf4) on a 64 x 64 sample of the output, from both the
    single-SM kernel and the CTA-pair kernel the benchmark's MXFP4 figure
    times; the two outputs are also equal byte for byte in full."""
    import torch
    a = _rand_bf16((M, D), 1.0, 101)
    b = _rand_bf16((H, D), 0.02, 102)
    ar, _, _ = cuda_lib.mx_quantize(a, O.E2M1, True, False)
    br, _, _ = cuda_lib.mx_quantize(b, O.E2M1, True, False)
    out = cuda_lib.mx_gemm_bias(ar, br, None)
    pair = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_2sm(ar, br, 1, None, out=pair)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    aq = _deq_rows(O.bf16_to_f64(_bits(a[_idx(ROWS)])), O.E2M1, False)
    bq = _deq_rows(O.bf16_to_f64(_bits(b[_idx(COLS)])), O.E2M1, False)
    for o in (out, pair):
        got = bf16_cpu(o[_idx(ROWS)][:, _idx(COLS)])
        assert O.within_tolerance(got, aq @ bq.T).all()
    assert torch.equal(out.view(torch.int16), pair.view(torch.int16))
