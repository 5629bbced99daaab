"""The training step captured in a CUDA graph and replayed.

mx_mlp_fwd_bwd enqueues its launches (and the weight gradients' counter
clears) asynchronously on the caller's stream, with no host synchronisation
unless MX_VALIDATE_OFFSETS is set and no allocation, so a caller can capture
the whole step once and replay it: the replays must give the eager step's
outputs bit for bit."""
import numpy as np
import pytest

import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_step_replayed_from_a_cuda_graph_equals_the_eager_step(cuda_lib, act):
    import torch
    mx = cuda_lib
    dev = "cuda"
    if act == "swiglu":
        G, D, F, R = 4, 512, 256, 1024
        inp = W.moe_inputs(G, D, F, R, seed=31)
        offs = torch.from_numpy(np.cumsum([384, 0, 256, 256]).astype(np.int32)).cuda()
        t = {k: to_dev(v) for k, v in inp.items()}
        out = {"y": torch.zeros((R, D), dtype=torch.bfloat16, device=dev),
               "dx": torch.zeros((R, D), dtype=torch.bfloat16, device=dev),
               "dw1": torch.zeros((G, 2 * F, D), dtype=torch.bfloat16, device=dev),
               "dw2": torch.zeros((G, D, F), dtype=torch.bfloat16, device=dev)}
        mk = lambda ws=None: mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], offs, G, F, out["y"], out["dx"],
                                         out["dw1"], out["dw2"], workspace=ws)
    else:
        M, D, H = 512, 256, 512
        inp = W.dense_inputs(M, D, H, seed=32)
        t = {k: to_dev(v) for k, v in inp.items()}
        out = {"y": torch.zeros((M, D), dtype=torch.bfloat16, device=dev),
               "dx": torch.zeros((M, D), dtype=torch.bfloat16, device=dev),
               "dw1": torch.zeros((H, D), dtype=torch.bfloat16, device=dev),
               "dw2": torch.zeros((D, H), dtype=torch.bfloat16, device=dev),
               "db1": torch.zeros(H, dtype=torch.float32, device=dev),
               "db2": torch.zeros(D, dtype=torch.float32, device=dev)}
        kw = dict(act=mx.ACT_GELU_TANH, fmt=mx.E2M3, hadamard=True, b1=t["b1"], b2=t["b2"], db1=out["db1"],
                  db2=out["db2"])
        mk = lambda ws=None: mx.mlp_args(t["x"], t["w1"], t["w2"], t["dy"], None, 1, H, out["y"], out["dx"],
                                         out["dw1"], out["dw2"], workspace=ws, **kw)
    ws = torch.empty(mx.mx_mlp_workspace_bytes(mk()), dtype=torch.uint8, device=dev)
    args = mk(ws)
    mx.mx_mlp_fwd_bwd(args)                     # eager step (also sets every kernel's launch attribute)
    torch.cuda.synchronize()
    assert mx.mx_get_device_status() == "MX_OK"
    eager = {k: v.clone() for k, v in out.items()}
    for v in out.values():
        v.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            mx.mx_mlp_fwd_bwd(args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for _ in range(2):
        for v in out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert mx.mx_get_device_status() == "MX_OK"
        for k in out:
            assert torch.equal(out[k], eager[k]), k
