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
from helpers import bf16_cpu, to_dev

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
    import torch
    counts, offsets, big, empty, small = routing
    x = _rand_bf16((R, D), 1.0, 11)
    w1 = _rand_bf16((G, 2 * F, D), 0.02, 12)
    offs = torch.from_numpy(offsets).cuda()
    xr, _, _ = cuda_lib.mx_quantize(x, O.E4M3, True, False)
    wr, _, _ = cuda_lib.mx_quantize(w1, O.E4M3, True, False)
    z, h_row, h_col = cuda_lib.mx_grouped_gemm_swiglu_fwd(xr, wr, G, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small, (big + 1) % G])
    xb = _bits(x[torch.from_numpy(rows).cuda()])
    zg = bf16_cpu(z[torch.from_numpy(rows).cuda()])
    hp = h_row.data[torch.from_numpy(rows).cuda()].cpu().numpy()
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        xq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(xb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w1[g])), O.E4M3), 2 * F, D, O.E4M3)
        zref = xq @ wq.T
        assert O.within_tolerance(zg[sel], zref).all(), g
        h = O.round_f32(O.swiglu(zref[:, :F], zref[:, F:]))
        ref_p, _ = O.quantize_rows(h, O.E4M3)
        assert np.mean(hp[sel] != ref_p) < 1e-2


def test_fc2_full_size_sampled_rows(cuda_lib, routing):
    import torch
    counts, offsets, big, empty, small = routing
    h = _rand_bf16((R, F), 0.5, 21)
    w2 = _rand_bf16((G, D, F), 0.02, 22)
    offs = torch.from_numpy(offsets).cuda()
    hr, _, _ = cuda_lib.mx_quantize(h, O.E4M3, True, False)
    w2r, _, _ = cuda_lib.mx_quantize(w2, O.E4M3, True, False)
    y = torch.full((R, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.mx_grouped_gemm(hr, w2r, G, offs, out=y)
    rows = _sample_rows(offsets, [big, small], seed=1)
    yg = bf16_cpu(y[torch.from_numpy(rows).cuda()])
    hb = _bits(h[torch.from_numpy(rows).cuda()])
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        hq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(hb[sel]), O.E4M3), int(sel.sum()), F, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2[g])), O.E4M3), D, F, O.E4M3)
        assert O.within_tolerance(yg[sel], hq @ wq.T).all(), g


def test_dswiglu_full_size_sampled_rows(cuda_lib, routing):
    import torch
    counts, offsets, big, empty, small = routing
    dy = _rand_bf16((R, D), 1e-3, 31)
    w2t = _rand_bf16((G, F, D), 0.02, 32)
    z = _rand_bf16((R, 2 * F), 2.0, 33)
    offs = torch.from_numpy(offsets).cuda()
    dyr, _, _ = cuda_lib.mx_quantize(dy, O.E4M3, True, False)
    wtr, _, _ = cuda_lib.mx_quantize(w2t, O.E4M3, True, False)
    dz_row, dz_col = cuda_lib.mx_grouped_gemm_dswiglu_bwd(dyr, wtr, z, G, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small], seed=2)
    idx = torch.from_numpy(rows).cuda()
    dzp = dz_row.data[idx].cpu().numpy()
    dyb, zb = _bits(dy[idx]), _bits(z[idx])
    for g in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == g for r in rows])
        dyq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(dyb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2t[g])), O.E4M3), F, D, O.E4M3)
        zf = O.bf16_to_f64(zb[sel])
        dg, du = O.dswiglu(dyq @ wq.T, zf[:, :F], zf[:, F:])
        ref_p, _ = O.quantize_rows(O.round_f32(np.concatenate([dg, du], axis=1)), O.E4M3)
        assert np.mean(dzp[sel] != ref_p) < 1e-2


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


def test_mlp_step_full_size_runs_and_is_deterministic(cuda_lib, routing):
    """The whole step at the benchmark's shape: status OK, finite outputs,
    zero gradient slices for empty experts, and bitwise repeatable."""
    import torch
    counts, offsets, big, empty, small = routing
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


def test_swiglu_probs_fwd_bwd_full_size_sampled_rows(cuda_lib, routing):
    """The routing-probability forms at full size: h = swiglu(z) * p[r]
    requantized (sampled rows within one step), and the backward's dz =
    dSwiGLU(dh * p) bytes and dprobs[r] = sum_f dh * swiglu(z) on the same
    rows (z saved by the forward, so the backward's input is the GPU's own
    BF16 z, which the oracle reads as given)."""
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
    z, h_row, _ = cuda_lib.mx_grouped_gemm_swiglu_probs_fwd(xr, wr, G, offs, probs)
    dyr, _, _ = cuda_lib.mx_quantize(dy, O.E4M3, True, False)
    wtr, _, _ = cuda_lib.mx_quantize(w2t, O.E4M3, True, False)
    dz_row, _, dprobs = cuda_lib.mx_grouped_gemm_dswiglu_probs_bwd(dyr, wtr, z, probs, G, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    rows = _sample_rows(offsets, [big, small], per=16, seed=5)
    idx = torch.from_numpy(rows).cuda()
    p = probs[idx].cpu().numpy().astype(np.float64)
    hp, dzp = h_row.data[idx].cpu().numpy(), dz_row.data[idx].cpu().numpy()
    dpg = dprobs[idx].cpu().numpy().astype(np.float64)
    xb, dyb, zb = _bits(x[idx]), _bits(dy[idx]), _bits(z[idx])
    for e in sorted({_expert_of(offsets, r) for r in rows}):
        sel = np.array([_expert_of(offsets, r) == e for r in rows])
        xq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(xb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        wq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w1[e])), O.E4M3), 2 * F, D, O.E4M3)
        zref = xq @ wq.T
        h = O.round_f32(O.swiglu(zref[:, :F], zref[:, F:]) * p[sel][:, None])
        assert np.mean(hp[sel] != O.quantize_rows(h, O.E4M3)[0]) < 1e-2
        dyq = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(dyb[sel]), O.E4M3), int(sel.sum()), D, O.E4M3)
        w2q = O.dequantize_rows(*O.quantize_rows(O.bf16_to_f64(_bits(w2t[e])), O.E4M3), F, D, O.E4M3)
        zf = O.bf16_to_f64(zb[sel])
        dh = dyq @ w2q.T
        act = O.swiglu(zf[:, :F], zf[:, F:])
        dg, du = O.dswiglu(dh * p[sel][:, None], zf[:, :F], zf[:, F:])
        ref_p, _ = O.quantize_rows(O.round_f32(np.concatenate([dg, du], axis=1)), O.E4M3)
        assert np.mean(dzp[sel] != ref_p) < 1e-2
        want = np.sum(dh * act, axis=1)
        scale = np.sqrt(np.sum((dh * act) ** 2, axis=1)) + 1e-30
        assert np.all(np.abs(dpg[sel] - want) <= 2.0 ** -8 * np.abs(want) + 2.0 ** -10 * scale), e


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
