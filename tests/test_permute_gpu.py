"""Token permute on the GPU against the oracle: the routing index bit for
bit, the quantizing permute's bytes (both orientations, three formats,
capacity rows past the routed segments untouched), the un-permute, and the
full-size routing (32768 tokens, top-8 of 128 experts) with sampled bytes."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import bf16_cpu, mx_bytes

pytestmark = pytest.mark.gpu


def _topk(rng, T, k, G, weights=None, skip=()):
    p = np.ones(G) if weights is None else np.asarray(weights, dtype=np.float64)
    p = p.copy()
    for e in skip:
        p[e] = 0.0
    p /= p.sum()
    return np.stack([rng.choice(G, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _route(mx, topk, G):
    import torch
    offs, src, row_of = mx.mx_moe_route_index(torch.from_numpy(topk).cuda(), G)
    assert mx.mx_get_device_status() == "MX_OK"
    return offs, src, row_of


@pytest.mark.parametrize("T,k,G", [(1000, 4, 8), (257, 1, 3), (3000, 8, 64)])
def test_route_index_bit_exact(cuda_lib, T, k, G):
    rng = np.random.default_rng(T + k)
    topk = _topk(rng, T, k, G, skip=(1,))
    offs, src, row_of = _route(cuda_lib, topk, G)
    r_off, r_src, r_row = O.moe_route_index(topk, G)
    R = int(r_off[-1])
    assert np.array_equal(offs.cpu().numpy(), r_off)
    s = src.cpu().numpy()
    assert np.array_equal(s[:R], r_src) and np.all(s[R:] == -1)
    assert np.array_equal(row_of.cpu().numpy(), r_row)
    assert src.numel() == cuda_lib.mx_moe_route_rows(T, k, G)


def test_route_index_out_of_range_expert_is_reported(cuda_lib):
    import torch
    topk = np.array([[0, 1], [2, 7], [1, 0]], dtype=np.int32)    # 7 >= G = 3
    offs, src, row_of = cuda_lib.mx_moe_route_index(torch.from_numpy(topk).cuda(), 3)
    assert cuda_lib.mx_get_device_status() == "MX_ERR_INVALID_ARG"
    assert row_of.cpu().numpy()[1, 1] == -1
    assert cuda_lib.mx_get_device_status() == "MX_OK"   # the report is cleared once read


def _compare_perm(mx, x_bits, topk, G, fmt, row, col, poison=True):
    import torch
    offs, src, _ = _route(mx, topk, G)
    R_cap = src.numel()
    D = x_bits.shape[1]
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    out_row = mx.MX(R_cap, D, fmt) if row else None
    out_col = mx.MX(D, R_cap, fmt) if col else None
    for t in (out_row, out_col):
        if t is not None and poison:
            t.data.fill_(0xA5)
            t.scale.fill_(0xA5)
    mx.mx_permute_quantize(x, src, offs, fmt=fmt, rowwise=row, colwise=col, out_row=out_row, out_col=out_col)
    assert mx.mx_get_device_status() == "MX_OK"
    r_off, r_src, _ = O.moe_route_index(topk, G)
    R = int(r_off[-1])
    ref = O.permute_quantize(x_bits, r_src, fmt, row, col)
    bpr = O.payload_row_bytes(D, fmt)
    if row:
        pay, sc = mx_bytes(out_row)
        assert np.array_equal(pay[:R], np.asarray(ref["row_payload"]).reshape(R, bpr))
        assert np.array_equal(O.scales_to_matrix(sc, R_cap, D // 32)[:R],
                              O.scales_to_matrix(ref["row_scales"], R, D // 32))
        if poison and R < R_cap:
            assert np.all(pay[R:] == 0xA5), "rows past the routed segments were written"
    if col:
        pay, sc = mx_bytes(out_col)
        cb = O.payload_row_bytes(R, fmt)
        assert np.array_equal(pay[:, :cb], np.asarray(ref["col_payload"]).reshape(D, cb))
        assert np.array_equal(O.scales_to_matrix(sc, D, R_cap // 32)[:, :R // 32],
                              O.scales_to_matrix(ref["col_scales"], D, R // 32))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M3, O.E2M1])
def test_permute_quantize_bytes(cuda_lib, fmt):
    rng = np.random.default_rng(90 + fmt)
    T, k, G, D = 1000, 4, 8, 256
    topk = _topk(rng, T, k, G, skip=(5,))
    x = W.normal_bf16(rng, (T, D))
    x[3, :] = 0                                        # a zero token: scale byte 0
    _compare_perm(cuda_lib, x, topk, G, fmt, True, True)


@pytest.mark.parametrize("row,col", [(True, False), (False, True)])
def test_permute_quantize_one_orientation(cuda_lib, row, col):
    rng = np.random.default_rng(95)
    T, k, G, D = 700, 2, 5, 384
    topk = _topk(rng, T, k, G)
    _compare_perm(cuda_lib, W.normal_bf16(rng, (T, D)), topk, G, O.E4M3, row, col)


def test_permute_quantize_rowwise_equals_gathered_token_quantization(cuda_lib):
    """The rowwise bytes of the permute equal the tokens' own rowwise
    quantization gathered by src (the quantize-before-permute identity),
    checked GPU against GPU."""
    import torch
    rng = np.random.default_rng(96)
    T, k, G, D = 512, 4, 8, 512
    topk = _topk(rng, T, k, G)
    offs, src, _ = _route(cuda_lib, topk, G)
    x = torch.from_numpy(W.normal_bf16(rng, (T, D)).view(np.int16)).cuda().view(torch.bfloat16)
    perm_row, _ = cuda_lib.mx_permute_quantize(x, src, offs, colwise=False)
    tok_row, _, _ = cuda_lib.mx_quantize(x, O.E4M3, True, False)
    s = src.cpu().numpy()
    R = int(offs[-1].item())
    pp, ps = mx_bytes(perm_row)
    tp, ts = mx_bytes(tok_row)
    used = s[:R] >= 0
    assert np.array_equal(pp[:R][used], tp[s[:R][used]])
    assert np.all(pp[:R][~used] == 0)
    psm = O.scales_to_matrix(ps, src.numel(), D // 32)[:R]
    tsm = O.scales_to_matrix(ts, T, D // 32)
    assert np.array_equal(psm[used], tsm[s[:R][used]]) and np.all(psm[~used] == 0)


def test_unpermute_against_oracle(cuda_lib):
    import torch
    rng = np.random.default_rng(97)
    T, k, G, D = 600, 4, 8, 256
    topk = _topk(rng, T, k, G)
    _, _, row_of = _route(cuda_lib, topk, G)
    r_off, _, r_row = O.moe_route_index(topk, G)
    R = int(r_off[-1])
    y_bits = W.normal_bf16(rng, (R, D))
    y = torch.from_numpy(y_bits.view(np.int16)).cuda().view(torch.bfloat16)
    w = rng.random((T, k)).astype(np.float32)
    out_w = cuda_lib.mx_moe_unpermute(y, row_of, torch.from_numpy(w).cuda())
    out_1 = cuda_lib.mx_moe_unpermute(y, row_of)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    yd = O.bf16_to_f64(y_bits)
    assert O.within_tolerance(bf16_cpu(out_w), O.unpermute(yd, r_row, w.astype(np.float64))).all()
    assert O.within_tolerance(bf16_cpu(out_1), O.unpermute(yd, r_row)).all()


def test_unpermute_exact_sums_bit_exact(cuda_lib):
    """Small-integer rows and power-of-two weights: every fp32 partial sum is
    exact, so the BF16 result is the oracle's rounding of the exact sum."""
    import torch
    rng = np.random.default_rng(98)
    T, k, G, D = 300, 8, 16, 128
    topk = _topk(rng, T, k, G)
    _, _, row_of = _route(cuda_lib, topk, G)
    r_off, _, r_row = O.moe_route_index(topk, G)
    R = int(r_off[-1])
    y = rng.integers(-40, 41, size=(R, D)).astype(np.float32)
    w = np.exp2(rng.integers(-3, 2, size=(T, k))).astype(np.float32)
    yt = torch.from_numpy(W.to_bf16_bits(y).view(np.int16)).cuda().view(torch.bfloat16)
    out = cuda_lib.mx_moe_unpermute(yt, row_of, torch.from_numpy(w).cuda())
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    assert np.array_equal(bf16_cpu(out), O.bf16_out(O.unpermute(y.astype(np.float64), r_row, w.astype(np.float64))))


def test_full_size_routing_and_sampled_permute_bytes(cuda_lib):
    """32768 tokens, top-8 of 128 experts (Zipf(1.1) expert popularity, one
    expert never chosen), D = 2048: the routing index bit for bit, and
    sampled routed rows (rowwise) and 32-row blocks (columnwise) of the
    quantizing permute against the oracle's quantization of those rows."""
    import torch
    rng = np.random.default_rng(99)
    T, k, G, D = 32768, 8, 128, 2048
    wts = 1.0 / np.arange(1, G + 1) ** 1.1
    topk = _topk(rng, T, k, G, weights=rng.permutation(wts), skip=(17,))
    offs, src, row_of = _route(cuda_lib, topk, G)
    r_off, r_src, r_row = O.moe_route_index(topk, G)
    R = int(r_off[-1])
    assert np.array_equal(offs.cpu().numpy(), r_off)
    assert np.array_equal(src.cpu().numpy()[:R], r_src)
    assert np.array_equal(row_of.cpu().numpy(), r_row)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn((T, D), generator=g, device="cuda").to(torch.bfloat16)
    out_row, out_col = cuda_lib.mx_permute_quantize(x, src, offs)
    assert cuda_lib.mx_get_device_status() == "MX_OK"
    xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
    prow, psc = mx_bytes(out_row)
    R_cap = src.numel()
    rows = rng.choice(R, size=64, replace=False)
    ref = O.quantize_bf16(O.permute_rows(xb, r_src[rows]), O.E4M3, True, False)
    assert np.array_equal(prow[rows], np.asarray(ref["row_payload"]).reshape(64, D))
    assert np.array_equal(O.scales_to_matrix(psc, R_cap, D // 32)[rows],
                          O.scales_to_matrix(ref["row_scales"], 64, D // 32))
    pcol, csc = mx_bytes(out_col)
    cs = O.scales_to_matrix(csc, D, R_cap // 32)
    for blk in rng.choice(R // 32, size=8, replace=False):
        ref = O.quantize_bf16(O.permute_rows(xb, r_src[blk * 32:(blk + 1) * 32]), O.E4M3, False, True)
        assert np.array_equal(pcol[:, blk * 32:(blk + 1) * 32], np.asarray(ref["col_payload"]).reshape(D, 32))
        assert np.array_equal(cs[:, blk], O.scales_to_matrix(ref["col_scales"], D, 1)[:, 0])
