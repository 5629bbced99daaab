"""Pins of the oracle's token permute / un-permute (CPU only), each against
something other than the oracle's own code: a hand-derived routing, the
counting-sort invariants, the exact commutation of rowwise MX quantization
with a row gather, and the adjoint identity between permute and
un-permute."""
import numpy as np
import pytest

import oracle as O
import workloads as W


def _topk(rng, T, k, G, skip=()):
    """k distinct experts per token (as a top-k router picks), never one in skip."""
    allowed = np.array([e for e in range(G) if e not in skip])
    return np.stack([rng.choice(allowed, size=k, replace=False) for _ in range(T)]).astype(np.int32)


def test_route_index_hand_example():
    """T=3 tokens, top-2 over 3 experts, segments padded to 4 rows:
    expert 0 gets (t0,j1), (t1,j0); expert 1 (t1,j1), (t2,j1); expert 2
    (t0,j0), (t2,j0) -- worked out by hand from the definition."""
    offsets, src, row_of = O.moe_route_index(np.array([[2, 0], [0, 1], [2, 1]]), 3, pad=4)
    assert offsets.tolist() == [4, 8, 12]
    assert src.tolist() == [0, 1, -1, -1, 1, 2, -1, -1, 0, 2, -1, -1]
    assert row_of.tolist() == [[8, 0], [1, 4], [9, 5]]


def test_route_index_empty_expert_and_single_choice():
    offsets, src, row_of = O.moe_route_index(np.array([[1], [1], [3]]), 4, pad=2)
    assert offsets.tolist() == [0, 2, 2, 4]        # experts 0 and 2 empty
    assert src.tolist() == [0, 1, 2, -1]
    assert row_of.ravel().tolist() == [0, 1, 2]


def test_route_index_rejects_out_of_range():
    with pytest.raises(ValueError):
        O.moe_route_index(np.array([[0, 5]]), 4)


@pytest.mark.parametrize("T,k,G", [(300, 4, 8), (1000, 8, 16)])
def test_route_index_invariants(T, k, G):
    """Counting-sort invariants: each (token, choice) lands on exactly one
    row holding its token, inside its expert's segment; segments are
    128-row multiples holding exactly the expert's count; within a segment
    tokens ascend; the rest of the segment is padding."""
    rng = np.random.default_rng(T)
    topk = _topk(rng, T, k, G, skip=(G // 2,))
    offsets, src, row_of = O.moe_route_index(topk, G)
    counts = np.bincount(topk.ravel(), minlength=G)
    segs = O.segments(offsets)
    assert all((e - s) % 128 == 0 and (e - s) == -(-counts[g] // 128) * 128 for g, (s, e) in enumerate(segs))
    assert counts[G // 2] == 0 and segs[G // 2][0] == segs[G // 2][1]
    assert sorted(row_of.ravel().tolist()) == sorted(np.nonzero(src >= 0)[0].tolist())
    assert np.all(src[row_of] == np.arange(T)[:, None])
    for g, (s, e) in enumerate(segs):
        seg = src[s:e]
        used = seg[: counts[g]]
        assert np.all(used >= 0) and np.all(np.diff(used) > 0) and np.all(seg[counts[g]:] == -1)
        assert np.all(np.any(topk[used] == g, axis=1))


def test_rowwise_quantization_commutes_with_the_gather():
    """Rowwise MX blocks lie inside one row, so quantizing the permuted rows
    gives exactly the gathered rowwise quantization of the tokens (the
    page's bit-identity of quantize-then-permute holds for MX rowwise blocks;
    columnwise blocks span 32 routed rows, so those are quantized in the
    permuted order)."""
    rng = np.random.default_rng(5)
    T, k, G, D = 200, 2, 4, 128
    topk = _topk(rng, T, k, G)
    _, src, _ = O.moe_route_index(topk, G)
    x = W.normal_bf16(rng, (T, D))
    perm = O.permute_quantize(x, src)
    tok = O.quantize_bf16(x, O.E4M3, True, False)
    R = len(src)
    pay = np.asarray(tok["row_payload"]).reshape(T, -1)
    sc = O.scales_to_matrix(tok["row_scales"], T, D // 32)
    want_pay = np.where((src >= 0)[:, None], pay[np.maximum(src, 0)], 0)
    want_sc = np.where((src >= 0)[:, None], sc[np.maximum(src, 0)], 0)
    assert np.array_equal(np.asarray(perm["row_payload"]).reshape(R, -1), want_pay)
    assert np.array_equal(O.scales_to_matrix(perm["row_scales"], R, D // 32), want_sc)


def test_unpermute_is_the_adjoint_of_permute():
    """<permute(x), y> = <x, unpermute(y)> for every x, y: pins the
    direction of both maps (a transposed index fails it)."""
    rng = np.random.default_rng(6)
    T, k, G, D = 150, 3, 5, 8
    topk = _topk(rng, T, k, G)
    _, src, row_of = O.moe_route_index(topk, G)
    x = rng.standard_normal((T, D))
    y = rng.standard_normal((len(src), D))
    lhs = np.sum(O.permute_rows(x, src) * y)
    rhs = np.sum(x * O.unpermute(y, row_of))
    assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + 1)


def test_unpermute_of_permute_scales_by_the_weight_sum():
    rng = np.random.default_rng(7)
    T, k, G, D = 64, 4, 6, 16
    topk = _topk(rng, T, k, G)
    _, src, row_of = O.moe_route_index(topk, G)
    x = rng.standard_normal((T, D))
    w = rng.random((T, k))
    assert np.allclose(O.unpermute(O.permute_rows(x, src), row_of), k * x, rtol=0, atol=1e-12)
    assert np.allclose(O.unpermute(O.permute_rows(x, src), row_of, w), w.sum(1)[:, None] * x, rtol=0, atol=1e-12)
