"""Full-size parity in the benchmark's launch configuration, on sampled outputs.

The MoE expert-MLP shape (G=128, D=2048, F=768, R=262144, Zipf(1.1) routing
with 8 empty experts) runs through the same persistent kernels the benchmark
times; the oracle recomputes sampled rows, column blocks and weight-gradient
entries one by one from the BF16 inputs.  Each stage gets its own seeded
BF16 inputs, so no oracle input ever comes from the CUDA path."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import assert_tap_requant_exact_sampled, bf16_cpu, decode_lut, mx_row_scales as mx_rows_scales, mx_rows_f64, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

G, D, F, R = W.MOE_SHAPE["G"], W.MOE_SHAPE["D"], W.MOE_SHAPE["F"], W.MOE_SHAPE["R"]


@pytest.fixture(scope="module")
def routing():
    counts = W.zipf_counts(G, R)
    offsets = W.offsets_from_counts(counts)
    big = int(np.argmax(counts))
    empty = int(np.flatnonzero(counts == 0)[0])
    small = int(np.flatnonzero(counts == counts[counts > 0].min())[0])
    return counts, offsets, big, empty, small


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _rand_bf16(shape, std, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16)


def _sample_rows(offsets, experts, per=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for g in experts:
        s, e = (int(offsets[g - 1]) if g else 0), int(offsets[g])
        if e > s:
            rows.extend(rng.choice(np.arange(s, e), size=min(per, e - s), replace=False).tolist())
    return np.array(sorted(rows))


def _expert_of(offsets, r):
    return int(np.searchsorted(offsets, r, side="right"))


def test_fc1_swiglu_full_size_sampled_rows(cuda_lib, routing):
    """FC1 + SwiGLU at full size with the debug tap attached: z and the
    epilogue's fp32 h within tolerance of the oracle on sampled rows of the
    largest, a small and a neighbouring expert, and both requantized
    orientations (payload and scale bytes) equal to the oracle's
    quantization of those fp32 values on the sampled rows and their 32-row
    column blocks."""
    import torch
    counts, offsets, big, empty, small = routing
    x = _rand_bf16((R, D), 1.0, 11)
    w1 = _rand_bf16((G, 2 * F, D), 0.02, 12)
    offs = torch.from_numpy(offsets).cuda()
    xr, _, _ = cuda_lib.mx_quantize(x, O.E4M3, True, False)
    wr, _, _ = cuda_lib.mx_quantize(w1, O.E4M3, True, False)
    tap = torch.full((R, F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap)
    try:
        z, h_row, h_col = cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, offs)
    finally:
        cuda_lib.mx_debug_tap(None)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small, (big + 1) % G])
    xb = _bits(x[torch.from_numpy(rows).cuda()])
    zg = bf16_cpu(z[torch.from_numpy(rows).cuda()])
    hg = tap[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        xq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(xb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w1[g])), O.E4M3), 2 * F, D, O.E4M3)
        zref = xq @ wq.T
        assert O.within_tolerance(zg[sel], zref).all(), g
        assert O.within_tolerance(hg[sel], O.round_f32(O.swiglu(zref[:, :F], zref[:, F:]))).all(), g
    assert_tap_requant_exact_sampled(h_row, h_col, tap, rows, what="h")


def test_fc2_full_size_sampled_rows(cuda_lib, routing):
    """FC2 at full size on one SM per tile and on CTA pairs: the two outputs
    byte-equal, and sampled rows of the largest and a small expert within
    tolerance of the oracle."""
    import torch
    counts, offsets, big, empty, small = routing
    h = _rand_bf16((R, F), 0.5, 21)
    w2 = _rand_bf16((G, D, F), 0.02, 22)
    offs = torch.from_numpy(offsets).cuda()
    hr, _, _ = cuda_lib.mx_quantize(h, O.E4M3, True, False)
    w2r, _, _ = cuda_lib.mx_quantize(w2, O.E4M3, True, False)
    y = torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(hr, w2r, G, offs, out=y)
    # the same product on CTA pairs (the kernel the step runs FC2 on)
    y2 = torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm_2sm(hr, w2r, G, offs, out=y2)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    A = int(offsets[-1])
    assert torch.equal(y[:A].view(torch.int16), y2[:A].view(torch.int16))
    rows = _sample_rows(offsets, [big, small], seed=1)
    hb = _bits(h[torch.from_numpy(rows).cuda()])
    for out in (y, y2):
        yg = bf16_cpu(out[torch.from_numpy(rows).cuda()])
        for g in sorted({_expert_of(offsets, r) for r in rows}):
            sel = np.array([_expert_of(offsets, r) == g for r in rows])
            hq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(hb[sel]), O.E4M3), int(sel.sum()), F, O.E4M3)
            wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2[g])), O.E4M3), D, F, O.E4M3)
            assert O.within_tolerance(yg[sel], hq @ wq.T).all(), g


def test_dswiglu_full_size_sampled_rows(cuda_lib, routing):
    """FC2 dgrad + dSwiGLU at full size with the debug tap attached: the
    epilogue's fp32 dz within tolerance of the oracle's dSwiGLU of the
    sampled rows' dh and saved z, and both requantized orientations equal to
    the oracle's quantization of those values."""
    import torch
    counts, offsets, big, empty, small = routing
    dy = _rand_bf16((R, D), 1e-3, 31)
    w2t = _rand_bf16((G, F, D), 0.02, 32)
    z = _rand_bf16((R, 2 * F), 2.0, 33)
    offs = torch.from_numpy(offsets).cuda()
    dyr, _, _ = cuda_lib.mx_quantize(dy, O.E4M3, True, False)
    wtr, _, _ = cuda_lib.mx_quantize(w2t, O.E4M3, True, False)
    tap = torch.full((R, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap)
    try:
        dz_row, dz_col = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, wtr, z, G, offs)
    finally:
        cuda_lib.mx_debug_tap(None)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small], seed=2)
    idx = torch.from_numpy(rows).cuda()
    dzg = tap[idx].cpu().numpy().astype(np.float64)
    dyb, zb = _bits(dy[idx]), _bits(z[idx])
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        dyq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(dyb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2t[g])), O.E4M3), F, D, O.E4M3)
        zf = O.bf16_to_f64(zb[sel])
        dg, du = O.dswiglu(dyq @ wq.T, zf[:, :F], zf[:, F:])
        assert O.within_tolerance(dzg[sel], O.round_f32(np.concatenate([dg, du], axis=1))).all(), g
    assert_tap_requant_exact_sampled(dz_row, dz_col, tap, rows, what="dz")


def test_wgrad_full_size_sampled_entries(cuda_lib, routing):
    """dW2[g] = dY_g^T h_g for the largest, a small and an empty expert:
    sampled entries recomputed from the BF16 columns of the segment, for
    the plain call and the K-split one the step uses."""
    import torch
    counts, offsets, big, empty, small = routing
    dy = _rand_bf16((R, D), 1e-3, 41)
    h = _rand_bf16((R, F), 0.5, 42)
    offs = torch.from_numpy(offsets).cuda()
    _, dyc, _ = cuda_lib.mx_quantize(dy, O.E4M3, False, True)
    _, hc, _ = cuda_lib.mx_quantize(h, O.E4M3, False, True)
    dw = cuda_lib.mx_grouped_gemm_wgrad(dyc, hc, G, offs)
    dws = cuda_lib.mx_grouped_gemm_wgrad_ws(dyc, hc, G, offs)   # the largest expert's K range split
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert bool((dw[empty] == 0).all()) and bool((dws[empty] == 0).all())
    rng = np.random.default_rng(4)
    for g in (big, small):
        s, e = int(offsets[g - 1]) if g else 0, int(offsets[g])
        ns = rng.choice(D, size=8, replace=False)
        a = O.bf16_to_f64(_bits(dy[s:e][:, torch.from_numpy(ns).cuda()]))   # [len, 8]
        b = O.bf16_to_f64(_bits(h[s:e]))                                    # [len, F]
        # columnwise quantization over the segment's 32-row blocks
        aq = O.dequantize_rows(*O.quantize_cols(a, O.E4M3), 8, e - s, O.E4M3)
        bq = O.dequantize_rows(*O.quantize_cols(b, O.E4M3), F, e - s, O.E4M3)
        ref = aq @ bq.T                                                     # 8 full rows of dW2[g]
        for out in (dw, dws):
            got = bf16_cpu(out[g][torch.from_numpy(ns).cuda()])
            assert O.within_tolerance(got, ref).all(), g


def _expert_rows(g, n):
    return np.arange(g * n, (g + 1) * n)


def test_mlp_step_full_size_sampled_parity(cuda_lib, routing):
    """The whole step at the benchmark's shape: status OK, bitwise
    repeatable, zero gradient slices for empty experts, and every stage held
    element by element to the oracle on the step's own intermediates (read
    back from its workspace) at sampled rows of the largest and a small
    expert: quantizer bytes exact; z, y, dX within tolerance; the fused
    requant bytes of h and dz equal the oracle's quantization of the
    epilogue's fp32 values (the stage re-run on the step's operands with the
    debug tap, giving the step's bytes); sampled dW1 / dW2 entries within
    tolerance."""
    import torch
    counts, offsets, big, empty, small = routing
    E = O.E4M3
    inp = W.moe_inputs_device(G, D, F, R, device="cuda")
    offs = torch.from_numpy(offsets).cuda()
    out = {"y": torch.empty((R, D), dtype=torch.bfloat16, device="cuda"),
           "dx": torch.empty((R, D), dtype=torch.bfloat16, device="cuda"),
           "dw1": torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device="cuda"),
           "dw2": torch.empty((G, D, F), dtype=torch.bfloat16, device="cuda")}
    a0 = cuda_lib.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                           out["dw2"])
    ws = torch.empty(cuda_lib.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device="cuda")
    args = cuda_lib.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], offs, G, F, out["y"], out["dx"],
                             out["dw1"], out["dw2"], workspace=ws)
    cuda_lib.mx_mlp_fwd_bwd(args)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    first = {k: v.clone() for k, v in out.items()}
    cuda_lib.mx_mlp_fwd_bwd(args)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    for k in out:
        assert torch.equal(first[k], out[k]), k
        assert bool(torch.isfinite(out[k].float()).all()), k
    assert bool((out["dw1"][empty] == 0).all()) and bool((out["dw2"][empty] == 0).all())
    del first
    V = cuda_lib.mlp_workspace_views(args, ws)
    lut = decode_lut(E)
    rows = _sample_rows(offsets, [big, small], per=8, seed=9)
    idx = torch.from_numpy(rows).cuda()

    # quantizers: sampled rows (rowwise) and their 32-row blocks (columnwise) exact
    for name in ("x", "dy"):
        src = inp[name]
        rp, rs = O.quantize_rows(O.bf16_to_f64(_bits(src[idx])), E)
        assert np.array_equal(V[name + "_row"].data[idx].cpu().numpy(), rp), name
        assert np.array_equal(mx_rows_scales(V[name + "_row"], rows), O.scales_to_matrix(rs, len(rows), D // 32)), name
        col_scales = mx_rows_scales(V[name + "_col"], np.arange(D))
        for b in np.unique(rows // 32):
            cp, cs = O.quantize_cols(O.bf16_to_f64(_bits(src[32 * b:32 * b + 32])), E)
            assert np.array_equal(V[name + "_col"].data[:, 32 * b:32 * b + 32].cpu().numpy(), cp), (name, b)
            assert np.array_equal(col_scales[:, b], O.scales_to_matrix(cs, D, 1)[:, 0]), (name, b)
    for g in (big, small):
        for name, n_rows, src, col in (("w1_row", 2 * F, inp["w1"][g], False), ("w1t_row", D, inp["w1"][g], True),
                                       ("w2_row", D, inp["w2"][g], False), ("w2t_row", F, inp["w2"][g], True)):
            q = (O.quantize_cols if col else O.quantize_rows)(O.bf16_to_f64(_bits(src)), E)
            er = _expert_rows(g, n_rows)
            m = V[name]
            assert np.array_equal(m.data[torch.from_numpy(er).cuda()].cpu().numpy(), q[0]), (name, g)
            assert np.array_equal(mx_rows_scales(m, er), O.scales_to_matrix(q[1], n_rows, m.cols // 32)), (name, g)

    # FC1 + SwiGLU, FC2 on sampled rows, from the step's own operands
    tap = torch.full((R, F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap)
    try:
        z2, h2r, h2c = cuda_lib.mx_grouped_gemm_swiglu_fwd(V["x_row"], V["w1_row"], G, offs)
    finally:
        cuda_lib.mx_debug_tap(None)
    A = int(offsets[-1])
    assert torch.equal(z2[:A], V["z"][:A]) and torch.equal(h2r.data[:A], V["h_row"].data[:A])
    assert torch.equal(h2c.data[:, :A], V["h_col"].data[:, :A])
    del z2, h2r, h2c
    assert_tap_requant_exact_sampled(V["h_row"], V["h_col"], tap, rows, what="h")
    zg = bf16_cpu(V["z"][idx])
    hg = tap[idx].cpu().numpy().astype(np.float64)
    del tap
    yg, dxg = bf16_cpu(out["y"][idx]), bf16_cpu(out["dx"][idx])
    dzrows = {}
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        xq = mx_rows_f64(V["x_row"], rows[sel], lut)
        w1q = mx_rows_f64(V["w1_row"], _expert_rows(g, 2 * F), lut)
        zref = xq @ w1q.T
        assert O.within_tolerance(zg[sel], zref).all(), ("z", g)
        assert O.within_tolerance(hg[sel], O.round_f32(O.swiglu(zref[:, :F], zref[:, F:]))).all(), ("h", g)
        yref = mx_rows_f64(V["h_row"], rows[sel], lut) @ mx_rows_f64(V["w2_row"], _expert_rows(g, D), lut).T
        assert O.within_tolerance(yg[sel], yref).all(), ("y", g)
        dh = mx_rows_f64(V["dy_row"], rows[sel], lut) @ mx_rows_f64(V["w2t_row"], _expert_rows(g, F), lut).T
        zf = O.bf16_to_f64(_bits(V["z"][torch.from_numpy(rows[sel]).cuda()]))
        dg, du = O.dswiglu(dh, zf[:, :F], zf[:, F:])
        dzrows[g] = (sel, O.round_f32(np.concatenate([dg, du], axis=1)))
        dxref = mx_rows_f64(V["dz_row"], rows[sel], lut) @ mx_rows_f64(V["w1t_row"], _expert_rows(g, D), lut).T
        assert O.within_tolerance(dxg[sel], dxref).all(), ("dx", g)

    # FC2 dgrad + dSwiGLU from the step's own dY, W2^T and z
    tap = torch.full((R, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap)
    try:
        d2r, d2c = cuda_lib.mx_grouped_gemm_dswiglu_bwd(V["dy_row"], V["w2t_row"], V["z"], G, offs)
    finally:
        cuda_lib.mx_debug_tap(None)
    assert torch.equal(d2r.data[:A], V["dz_row"].data[:A]) and torch.equal(d2c.data[:, :A], V["dz_col"].data[:, :A])
    del d2r, d2c
    assert_tap_requant_exact_sampled(V["dz_row"], V["dz_col"], tap, rows, what="dz")
    dzg = tap[idx].cpu().numpy().astype(np.float64)
    del tap
    for g, (sel, dzref) in dzrows.items():
        assert O.within_tolerance(dzg[sel], dzref).all(), ("dz", g)

    # weight gradients: sampled entries of the largest and a small expert
    rng = np.random.default_rng(10)
    for g in (big, small):
        s, e = (int(offsets[g - 1]) if g else 0), int(offsets[g])
        for name, a_name, b_name, n_a, n_b in (("dw2", "dy_col", "h_col", D, F), ("dw1", "dz_col", "x_col", 2 * F, D)):
            ns, ks = np.sort(rng.choice(n_a, 8, replace=False)), np.sort(rng.choice(n_b, 8, replace=False))
            aq = mx_rows_f64(V[a_name], ns, lut)[:, s:e]
            bq = mx_rows_f64(V[b_name], ks, lut)[:, s:e]
            got = bf16_cpu(out[name][g][torch.from_numpy(ns).cuda()][:, torch.from_numpy(ks).cuda()])
            assert O.within_tolerance(got, aq @ bq.T).all(), (name, g)


def test_swiglu_probs_fwd_bwd_full_size_sampled_rows(cuda_lib, routing):
    """The routing-probability forms at full size with the debug tap
    attached: the forward's fp32 h = swiglu(z) * p[r] and the backward's fp32
    dz = dSwiGLU(dh * p) within tolerance of the oracle on sampled rows, both
    requantized orientations (payload and scale bytes) equal to the oracle's
    quantization of those fp32 values, and dprobs[r] = sum_f dh * swiglu(z)
    on the same rows (z saved by the forward, so the backward's input is the
    GPU's own BF16 z, which the oracle reads as given)."""
    import torch
    counts, offsets, big, empty, small = routing
    x = _rand_bf16((R, D), 1.0, 111)
    w1 = _rand_bf16((G, 2 * F, D), 0.02, 112)
    dy = _rand_bf16((R, D), 1e-3, 113)
    w2t = _rand_bf16((G, F, D), 0.02, 114)
    g = torch.Generator(device="cuda")
    g.manual_seed(115)
    probs = torch.rand(R, generator=g, device="cuda") * 0.9 + 0.05
    offs = torch.from_numpy(offsets).cuda()
    xr, _, _ = cuda_lib.mx_quantize(x, O.E4M3, True, False)
    wr, _, _ = cuda_lib.mx_quantize(w1, O.E4M3, True, False)
    tap_h = torch.full((R, F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap_h)
    try:
        z, h_row, h_col = cuda_lib.mx_grouped_gemm_swiglu_probs_fwd(xr, wr, G, offs, probs)
    finally:
        cuda_lib.mx_debug_tap(None)
    dyr, _, _ = cuda_lib.mx_quantize(dy, O.E4M3, True, False)
    wtr, _, _ = cuda_lib.mx_quantize(w2t, O.E4M3, True, False)
    tap_dz = torch.full((R, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.mx_debug_tap(tap_dz)
    try:
        dz_row, dz_col, dprobs = cuda_lib.mx_grouped_gemm_dswiglu_probs_bwd(dyr, wtr, z, probs, G, offs)
    finally:
        cuda_lib.mx_debug_tap(None)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small], per=16, seed=5)
    idx = torch.from_numpy(rows).cuda()
    p = probs[idx].cpu().numpy().astype(np.float64)
    hg = tap_h[idx].cpu().numpy().astype(np.float64)
    dzg = tap_dz[idx].cpu().numpy().astype(np.float64)
    dpg = dprobs[idx].cpu().numpy().astype(np.float64)
    xb, dyb, zb = _bits(x[idx]), _bits(dy[idx]), _bits(z[idx])
    for e in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == e for r in rows])
        xq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(xb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w1[e])), O.E4M3), 2 * F, D, O.E4M3)
        zref = xq @ wq.T
        h = O.round_f32(O.swiglu(zref[:, :F], zref[:, F:]) * p[sel][:, None])
        assert O.within_tolerance(hg[sel], h).all(), e
        dyq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(dyb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        w2q = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2t[e])), O.E4M3), F, D, O.E4M3)
        zf = O.bf16_to_f64(zb[sel])
        dh = dyq @ w2q.T
        act = O.swiglu(zf[:, :F], zf[:, F:])
        dg, du = O.dswiglu(dh * p[sel][:, None], zf[:, :F], zf[:, F:])
        assert O.within_tolerance(dzg[sel], O.round_f32(np.concatenate([dg, du], axis=1))).all(), e
        want = np.sum(dh * act, axis=1)
        # dprobs is one vector: the tolerance's "row" is the sampled vector
        assert O.within_tolerance(dpg[sel][None, :], want[None, :]).all(), e
    assert_tap_requant_exact_sampled(h_row, h_col, tap_h, rows, what="h * p")
    assert_tap_requant_exact_sampled(dz_row, dz_col, tap_dz, rows, what="dSwiGLU(dh * p)")


def test_wgrad_into_fp32_full_size_sampled_entries(cuda_lib, routing):
    """The fp32 main-grad wgrad at full size (largest expert, K-split form):
    the store within tolerance of the oracle's entries, the accumulate equal
    to grad + store bit for bit, an empty expert's slice zero / untouched."""
    import torch
    counts, offsets, big, empty, small = routing
    dy = _rand_bf16((R, D), 1e-3, 121)
    h = _rand_bf16((R, F), 0.5, 122)
    offs = torch.from_numpy(offsets).cuda()
    _, dyc, _ = cuda_lib.mx_quantize(dy, O.E4M3, False, True)
    _, hc, _ = cuda_lib.mx_quantize(h, O.E4M3, False, True)
    st = torch.empty((G, D, F), dtype=torch.float32, device="cuda")
    cuda_lib.mx_grouped_gemm_wgrad_f32_ws(dyc, hc, G, offs, st, accumulate=False)
    g0 = _rand_bf16((G, D, F), 1e-2, 123).float()
    acc = g0.clone()
    cuda_lib.mx_grouped_gemm_wgrad_f32_ws(dyc, hc, G, offs, acc, accumulate=True)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert bool((st[empty] == 0).all()) and torch.equal(acc[empty], g0[empty])
    assert torch.equal(acc, g0 + st), "accumulate is not fl32(grad + the stored sum)"
    rng = np.random.default_rng(6)
    s, e = (int(offsets[big - 1]) if big else 0), int(offsets[big])
    ns, ks = np.sort(rng.choice(D, 8, replace=False)), np.sort(rng.choice(F, 8, replace=False))
    a = O.bf16_to_f64(_bits(dy[s:e][:, torch.from_numpy(ns).cuda()]))
    b = O.bf16_to_f64(_bits(h[s:e][:, torch.from_numpy(ks).cuda()]))
    aq = O.dequantize_rows(*O.quantize_cols(a, O.E4M3), 8, e - s, O.E4M3)
    bq = O.dequantize_rows(*O.quantize_cols(b, O.E4M3), 8, e - s, O.E4M3)
    got = st[big][torch.from_numpy(ns).cuda()][:, torch.from_numpy(ks).cuda()].cpu().numpy().astype(np.float64)
    assert O.within_tolerance(got, aq @ bq.T).all()
