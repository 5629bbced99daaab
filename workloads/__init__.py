"""Seeded synthetic inputs for the MX training-MLP path.

Shared by the tests, the benchmark and the smoke check.  It holds no
arithmetic of the method (no quantization, no GEMM, no activation): only
random draws, their conversion to BF16 storage, and routing layouts.

Recipes (the pages' workloads are training data and model weights that are
not available; these stand in for their shapes and value distributions):

* ``pr_ref``            X, W BF16 [256, 256] ~ N(0, 1), seed 0, X drawn first.
* ``quantizer_input``   BF16 [8192, 7168]: t(df=3) * 2^u_row, u_row ~ U(-20, 20)
                        per row, seed 0, with 0.1 % of positions replaced by
                        specials drawn equally from {+0, -0, +Inf, -Inf, NaN,
                        BF16 subnormal, +-power of two >= its block's amax}.
* ``moe_inputs``        G experts, hidden D, FFN F, R routed rows: X ~ N(0, 1),
                        W1 [G, 2F, D] and W2 [G, D, F] ~ N(0, 0.02), seed 0,
                        drawn in the order X, W1, W2; dY ~ N(0, 1e-3), seed 2.
* ``even_offsets``      R/G rows per expert.
* ``zipf_offsets``      rank weights k^-s over ranks 1..G, 128-row tiles
                        floor(T * w_k / sum w), the n_zero lowest-weight ranks
                        forced to 0 tiles, leftover tiles to rank 1, ranks
                        mapped to expert ids by a seed-1 permutation.
* ``dense_inputs``      X [M, D] ~ N(0, 1), W1 [H, D], W2 [D, H], b1 [H],
                        b2 [D] ~ N(0, 0.02), dY [M, D] ~ N(0, 1e-3), seed 0.

Normal draws are float32 (numpy PCG64, Ziggurat), stored as BF16 by
round-to-nearest-even of the float32 bit pattern.
"""
import numpy as np

_CHUNK = 1 << 24


def to_bf16_bits(x):
    """float32 array -> BF16 bit patterns (uint16), nearest-even; NaN kept."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng, shape, std=1.0):
    """N(0, std^2) drawn in float32 chunks, stored as BF16 bits."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:e] = to_bf16_bits(v)
    return out.reshape(shape)


def pr_ref(n=256, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = normal_bf16(rng, (n, n))
    w = normal_bf16(rng, (n, n))
    return x, w


SPECIAL_KINDS = ("pos_zero", "neg_zero", "pos_inf", "neg_inf", "nan", "subnormal", "pow2_block_max")


def quantizer_input(rows=8192, cols=7168, seed=0, special_frac=0.001):
    """Heavy-tailed rows spanning 2^+-20 with injected special values."""
    rng = np.random.Generator(np.random.PCG64(seed))
    t = rng.standard_t(3, size=(rows, cols)).astype(np.float32)
    u = rng.uniform(-20.0, 20.0, size=(rows, 1))
    x = (t * np.exp2(u)).astype(np.float32)
    bits = to_bf16_bits(x)
    n = rows * cols
    k = int(round(special_frac * n))
    pos = rng.choice(n, size=k, replace=False)
    kinds = rng.integers(0, len(SPECIAL_KINDS), size=k)
    flat = bits.reshape(-1)
    vals = bf16_bits_to_f32(flat)
    for kind_id, name in enumerate(SPECIAL_KINDS):
        p = pos[kinds == kind_id]
        if name == "pos_zero":
            flat[p] = 0x0000
        elif name == "neg_zero":
            flat[p] = 0x8000
        elif name == "pos_inf":
            flat[p] = 0x7F80
        elif name == "neg_inf":
            flat[p] = 0xFF80
        elif name == "nan":
            flat[p] = 0x7FC0
        elif name == "subnormal":
            mant = rng.integers(1, 128, size=p.size).astype(np.uint16)
            sign = (rng.integers(0, 2, size=p.size).astype(np.uint16) << 15)
            flat[p] = sign | mant
        elif name == "pow2_block_max":
            # the smallest power of two >= the 32-column block's amax
            r, c = p // cols, p % cols
            c0 = (c // 32) * 32
            blk = np.abs(vals.reshape(rows, cols)[r[:, None], c0[:, None] + np.arange(32)[None, :]])
            amax = np.nanmax(np.where(np.isfinite(blk), blk, 0.0), axis=1)
            amax = np.maximum(amax, np.float32(2.0 ** -126))
            e = np.ceil(np.log2(amax.astype(np.float64)))
            e = np.clip(e, -126, 127)
            sign = np.where(rng.integers(0, 2, size=p.size) == 1, -1.0, 1.0)
            flat[p] = to_bf16_bits((sign * np.exp2(e)).astype(np.float32))
    return bits


def even_offsets(G, R):
    assert R % G == 0
    return (np.arange(1, G + 1, dtype=np.int64) * (R // G)).astype(np.int32)


def zipf_counts(G=128, R=262144, s=1.1, n_zero=8, seed=1, tile=128):
    T = R // tile
    ranks = np.arange(1, G + 1, dtype=np.float64)
    w = ranks ** (-s)
    t = np.floor(T * w / w.sum()).astype(np.int64)
    if n_zero:
        t[G - n_zero:] = 0
    t[0] += T - t.sum()
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(G)          # rank i -> expert perm[i]
    counts = np.zeros(G, dtype=np.int64)
    counts[perm] = t * tile
    return counts


def zipf_offsets(G=128, R=262144, s=1.1, n_zero=8, seed=1):
    return np.cumsum(zipf_counts(G, R, s, n_zero, seed)).astype(np.int32)


def offsets_from_counts(counts):
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


def moe_inputs(G, D, F, R, seed=0, dy_seed=2, with_dy=True):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = normal_bf16(rng, (R, D))
    w1 = normal_bf16(rng, (G, 2 * F, D), std=0.02)
    w2 = normal_bf16(rng, (G, D, F), std=0.02)
    out = {"x": x, "w1": w1, "w2": w2}
    if with_dy:
        rng2 = np.random.Generator(np.random.PCG64(dy_seed))
        out["dy"] = normal_bf16(rng2, (R, D), std=1e-3)
    return out


def dense_inputs(M, D, H, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return {
        "x": normal_bf16(rng, (M, D)),
        "w1": normal_bf16(rng, (H, D), std=0.02),
        "w2": normal_bf16(rng, (D, H), std=0.02),
        "b1": normal_bf16(rng, (H,), std=0.02),
        "b2": normal_bf16(rng, (D,), std=0.02),
        "dy": normal_bf16(rng, (M, D), std=1e-3),
    }


# The configurations the library is measured and checked on.
MOE_SHAPE = dict(G=128, D=2048, F=768, R=262144)
DENSE_SHAPE = dict(M=16384, D=3072, H=12288)
QUANT_SHAPE = dict(rows=8192, cols=7168)


def moe_inputs_device(G, D, F, R, seed=0, dy_seed=2, device="cuda"):
    """Full-size MoE inputs drawn on the GPU (same distributions as
    ``moe_inputs``; torch's seeded device generator, so the values differ
    from the numpy draw).  Used where drawing ~1.7e9 normals on the host
    would dominate the run."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((R, D), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    w1 = (torch.randn((G, 2 * F, D), generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((G, D, F), generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    g.manual_seed(dy_seed)
    dy = (torch.randn((R, D), generator=g, device=device, dtype=torch.float32) * 1e-3).to(torch.bfloat16)
    return {"x": x, "w1": w1, "w2": w2, "dy": dy}
