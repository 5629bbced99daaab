"""The no-allocation column-sum quantizer (mx_quantize_colsum_noalloc).

Some callers cannot allocate device memory at the point where they quantize
(a fixed memory pool, an embedding that owns all memory):
this entry point keeps its column-sum partials in a fixed scratch array
inside the library.  Its results must equal the workspace variant's, call
after call, since every call shares and rewrites the same scratch.

This file is collected last so that a failure here comes after every other
test has run."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,fmt,had", [(1024, 384, O.E2M3, True), (96, 160, O.E4M3, False)])
def test_noalloc_matches_workspace_variant_on_two_calls(cuda_lib, rows, cols, fmt, had):
    import torch
    bits = W.normal_bf16(np.random.default_rng(rows + cols), (rows, cols), std=1e-3)
    x = to_dev(bits)
    ref_row, ref_col, ref_cs = cuda_lib.mx_quantize(x, fmt, True, True, had, True)
    for _ in range(2):
        row, col, cs = cuda_lib.mx_quantize_colsum_noalloc(x, fmt, True, had)
        torch.cuda.synchronize()
        assert torch.equal(row.data, ref_row.data) and torch.equal(row.scale, ref_row.scale)
        assert torch.equal(col.data, ref_col.data) and torch.equal(col.scale, ref_col.scale)
        got, want = cs.cpu().numpy().astype(np.float64), ref_cs.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2.0 ** -14 * np.sqrt(np.mean(want ** 2)))
    # the sums themselves, against the oracle
    want = O.colsum(O.bf16_to_f64(bits))
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2.0 ** -14 * np.sqrt(np.mean(want ** 2)))


def test_noalloc_zero_rows_gives_zero_sums(cuda_lib):
    """No rows: nothing to quantize, and each column's sum over no rows is 0."""
    import torch
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    cs = torch.full((256,), float("nan"), dtype=torch.float32, device="cuda")
    _, _, cs = cuda_lib.mx_quantize_colsum_noalloc(x, O.E4M3, True, colsum_out=cs)
    torch.cuda.synchronize()
    assert bool((cs == 0).all())


def test_noalloc_rejects_sizes_beyond_the_scratch(cuda_lib):
    import torch
    rows, cols = 128 * 65, 32768          # 65 tile rows x 32768 columns > 2^21 partials
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.MXError) as e:
        cuda_lib.mx_quantize_colsum_noalloc(x, O.E4M3, False)
    assert e.value.name == "MX_ERR_WORKSPACE" and "scratch" in str(e.value)
