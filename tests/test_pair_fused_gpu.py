"""The fused SwiGLU forward, dSwiGLU backward and ragged-K weight gradient
on CTA pairs.

MX_FUSED_PAIRS=1 runs all three on CTA pairs (256-row tiles, .cta_group::2
MMAs; by default only the SwiGLU forward), MX_FUSED_PAIRS=0 keeps all on one
SM per tile.  The two are the same K order of block-scaled MMAs into fp32
and the same epilogue code, so every output byte must agree: the requantized
payloads and scales of both orientations, the BF16 pre-activation save, the
routing-probability gradient, the weight gradients (split or not) --
including segments with an odd number of 128-row blocks, whose last 256-row
tile computes an upper half that must not be stored, and a poisoned
inactive tail."""
import numpy as np
import pytest

import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu


def _inputs(mx, counts, F, D, seed, tail=256):
    import torch
    G = len(counts)
    offsets = W.offsets_from_counts(counts)
    R = int(offsets[-1]) + tail
    rng = np.random.default_rng(seed)
    x = to_dev(W.normal_bf16(rng, (R, D)))
    w1 = to_dev(W.normal_bf16(rng, (G, 2 * F, D), std=0.02))
    w2 = to_dev(W.normal_bf16(rng, (G, D, F), std=0.02))
    dy = to_dev(W.normal_bf16(rng, (R, D), std=1e-3))
    probs = torch.from_numpy(rng.uniform(0.05, 1.0, R).astype(np.float32)).cuda()
    xr, _, _ = mx.mx_quantize(x, mx.E4M3, True, False)
    w1r, _, _ = mx.mx_quantize(w1, mx.E4M3, True, False)
    _, w2t, _ = mx.mx_quantize(w2, mx.E4M3, False, True)
    dyr, _, _ = mx.mx_quantize(dy, mx.E4M3, True, False)
    return G, R, torch.from_numpy(offsets).cuda(), xr, w1r, w2t, dyr, probs


def _fill(t, byte):
    t.data.fill_(byte)
    t.scale.fill_(byte)


def _fwd(mx, G, R, F, offs, xr, w1r, probs, use_probs):
    import torch
    h_row, h_col = mx.MX(R, F), mx.MX(F, R)
    _fill(h_row, 0x5A)
    _fill(h_col, 0x5A)
    z = torch.full((R, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
    if use_probs:
        mx.mx_grouped_gemm_swiglu_probs_fwd(xr, w1r, G, offs, probs, h_row, h_col, z)
    else:
        mx.mx_grouped_gemm_swiglu_fwd(xr, w1r, G, offs, h_row, h_col, z)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    return [h_row.data, h_row.scale, h_col.data, h_col.scale, z]


def _bwd(mx, G, R, F, offs, dyr, w2t, z, probs, use_probs):
    import torch
    dz_row, dz_col = mx.MX(R, 2 * F), mx.MX(2 * F, R)
    _fill(dz_row, 0xA5)
    _fill(dz_col, 0xA5)
    out = [dz_row.data, dz_row.scale, dz_col.data, dz_col.scale]
    if use_probs:
        dprobs = torch.full((R,), float("nan"), dtype=torch.float32, device="cuda")
        mx.mx_grouped_gemm_dswiglu_probs_bwd(dyr, w2t, z, probs, G, offs, dz_row, dz_col, dprobs)
        out.append(dprobs)
    else:
        mx.mx_grouped_gemm_dswiglu_bwd(dyr, w2t, z, G, offs, dz_row, dz_col)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    return out


def _equal(a, b, names):
    import torch
    for x, y, n in zip(a, b, names):   # byte for byte (NaN fills compare equal)
        assert torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8)), \
            "%s differs between the pair and single-SM kernels" % n


@pytest.mark.parametrize("F,counts,use_probs", [
    (256, [384, 0, 128, 640], False),
    (512, [256, 256, 512], True),
    (768, [128, 896], False),
])
def test_fused_pairs_equal_single_sm(cuda_lib, monkeypatch, F, counts, use_probs):
    mx = cuda_lib
    D = 512
    G, R, offs, xr, w1r, w2t, dyr, probs = _inputs(mx, counts, F, D, seed=F + len(counts))
    monkeypatch.setenv("MX_FUSED_PAIRS", "1")
    fp = _fwd(mx, G, R, F, offs, xr, w1r, probs, use_probs)
    bp = _bwd(mx, G, R, F, offs, dyr, w2t, fp[4], probs, use_probs)
    monkeypatch.setenv("MX_FUSED_PAIRS", "0")
    fs = _fwd(mx, G, R, F, offs, xr, w1r, probs, use_probs)
    bs = _bwd(mx, G, R, F, offs, dyr, w2t, fs[4], probs, use_probs)
    _equal(fp, fs, ["h_row", "h_row scales", "h_col", "h_col scales", "z"])
    _equal(bp, bs, ["dz_row", "dz_row scales", "dz_col", "dz_col scales", "dprobs"])


@pytest.mark.parametrize("counts,ws,f32", [
    ([384, 0, 1920, 128, 640], False, False),   # one SM per tile's dealt order vs the pairs' (static)
    ([384, 0, 1920, 128, 640], True, False),    # claimed tiles and the largest expert's K range split
    ([256, 2816, 0, 512], True, True),          # fp32 store into main_grad, split
])
def test_wgrad_pairs_equal_single_sm(cuda_lib, monkeypatch, counts, ws, f32):
    """The ragged-K weight gradient on CTA pairs (256 x 256 tiles of the
    weight, the claimed-tile queue shared across the pair, each CTA's K-split
    partials in slots of their own) equals one SM per tile byte for byte,
    zero-token experts included."""
    import torch
    mx = cuda_lib
    G = len(counts)
    offsets = W.offsets_from_counts(counts)
    R = int(offsets[-1]) + 128
    N, K = 512, 768   # dW rows (a_col) and columns (b_col)
    rng = np.random.default_rng(len(counts) * 7 + (1 if ws else 0))
    a = to_dev(W.normal_bf16(rng, (R, N), std=1e-3))
    b = to_dev(W.normal_bf16(rng, (R, K)))
    _, a_col, _ = mx.mx_quantize(a, mx.E4M3, False, True)
    _, b_col, _ = mx.mx_quantize(b, mx.E4M3, False, True)
    offs = torch.from_numpy(offsets).cuda()

    def run():
        if f32:
            out = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
            if ws:
                mx.mx_grouped_gemm_wgrad_f32_ws(a_col, b_col, G, offs, out)
            else:
                mx.mx_grouped_gemm_wgrad_f32(a_col, b_col, G, offs, out)
        else:
            out = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
            if ws:
                mx.mx_grouped_gemm_wgrad_ws(a_col, b_col, G, offs, out=out)
            else:
                mx.mx_grouped_gemm_wgrad(a_col, b_col, G, offs, out=out)
        torch.cuda.synchronize()
        assert mx.mx_get_device_status() == "MX_OK"
        return out

    monkeypatch.setenv("MX_FUSED_PAIRS", "1")
    pair = run()
    monkeypatch.setenv("MX_FUSED_PAIRS", "0")
    single = run()
    _equal([pair], [single], ["dW"])
    empty = [g for g, c in enumerate(counts) if c == 0]
    for g in empty:   # a zero-token expert's slice is exactly zero
        assert bool((pair[g] == 0).all())
