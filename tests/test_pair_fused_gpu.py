"""The fused SwiGLU forward and dSwiGLU backward on CTA pairs.

MX_FUSED_PAIRS=1 runs both fused epilogues on CTA pairs (256-row tiles,
.cta_group::2 MMAs; by default only the SwiGLU forward), MX_FUSED_PAIRS=0
keeps both on one SM per tile.
The two are the same K order of block-scaled MMAs into fp32 and the same
epilogue code, so every output byte must agree: the requantized payloads and
scales of both orientations, the BF16 pre-activation save, the routing
probability gradient -- including segments with an odd number of 128-row
blocks, whose last 256-row tile computes an upper half that must not be
stored, and a poisoned inactive tail."""
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
