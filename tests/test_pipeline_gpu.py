"""The host-buffer pipeline (mx_mlp_pipeline_*): several steps enqueued back
to back, each with its own inputs, routing and host output buffers, must give
exactly what mx_mlp_fwd_bwd gives for the same inputs on device buffers (the
kernels are deterministic, so the comparison is bitwise).  Catches any copy
that overtakes the launch it is ordered against."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


def _pinned(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def _device_step(mx, inp, offs, G, F, act, fmt, had):
    """Reference: the step on device buffers, outputs copied to the CPU."""
    import torch
    dev = "cuda"
    R, D = inp["x"].shape
    F1 = 2 * F if act == mx.ACT_SWIGLU else F
    out = {"y": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
           "dx": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
           "dw1": torch.empty(inp["w1"].shape, dtype=torch.bfloat16, device=dev),
           "dw2": torch.empty(inp["w2"].shape, dtype=torch.bfloat16, device=dev)}
    extra = {}
    if act != mx.ACT_SWIGLU:
        out["db1"] = torch.empty(F1, dtype=torch.float32, device=dev)
        out["db2"] = torch.empty(D, dtype=torch.float32, device=dev)
        extra = dict(b1=inp["b1"].cuda(), b2=inp["b2"].cuda(), db1=out["db1"], db2=out["db2"])
    d = {k: inp[k].cuda() for k in ("x", "w1", "w2", "dy")}
    doff = offs.cuda() if offs is not None else None
    a0 = mx.mlp_args(d["x"], d["w1"], d["w2"], d["dy"], doff, G, F, out["y"], out["dx"], out["dw1"], out["dw2"],
                     act=act, fmt=fmt, hadamard=had, **extra)
    ws = torch.empty(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device=dev)
    a = mx.mlp_args(d["x"], d["w1"], d["w2"], d["dy"], doff, G, F, out["y"], out["dx"], out["dw1"], out["dw2"],
                    workspace=ws, act=act, fmt=fmt, hadamard=had, **extra)
    mx.mx_mlp_fwd_bwd(a)
    assert mx.mx_get_device_status() == "MX_OK"
    return {k: v.cpu() for k, v in out.items()}


def _pipeline_steps(mx, steps, G, F, act, fmt, had):
    """Run every step through one pipeline; returns the host outputs per step."""
    import torch
    dev = "cuda"
    inp0, _ = steps[0]
    R, D = inp0["x"].shape
    F1 = 2 * F if act == mx.ACT_SWIGLU else F
    dd = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in inp0.items()}
    dout = {"y": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "dx": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "dw1": torch.empty(inp0["w1"].shape, dtype=torch.bfloat16, device=dev),
            "dw2": torch.empty(inp0["w2"].shape, dtype=torch.bfloat16, device=dev)}
    extra = {}
    if act != mx.ACT_SWIGLU:
        dout["db1"] = torch.empty(F1, dtype=torch.float32, device=dev)
        dout["db2"] = torch.empty(D, dtype=torch.float32, device=dev)
        extra = dict(b1=dd["b1"], b2=dd["b2"], db1=dout["db1"], db2=dout["db2"])
    doff = torch.empty(G, dtype=torch.int32, device=dev) if steps[0][1] is not None else None
    a0 = mx.mlp_args(dd["x"], dd["w1"], dd["w2"], dd["dy"], doff, G, F, dout["y"], dout["dx"], dout["dw1"],
                     dout["dw2"], act=act, fmt=fmt, hadamard=had, **extra)
    ws = torch.empty(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device=dev)
    a = mx.mlp_args(dd["x"], dd["w1"], dd["w2"], dd["dy"], doff, G, F, dout["y"], dout["dx"], dout["dw1"],
                    dout["dw2"], workspace=ws, act=act, fmt=fmt, hadamard=had, **extra)
    pipe = mx.MlpPipeline(a)
    results = []
    host_keep = []
    for inp, offs in steps:
        host = {k: _pinned(v) for k, v in inp.items()}
        if offs is not None:
            host["offsets"] = _pinned(offs)
        outs = {k: torch.full(v.shape, float("nan"), dtype=v.dtype, pin_memory=True) for k, v in dout.items()}
        host.update(outs)
        pipe.run(host)
        host_keep.append(host)
        results.append(outs)
    pipe.sync()
    pipe.close()
    assert mx.mx_get_device_status() == "MX_OK"
    return results


def test_pipeline_swiglu_steps_match_device_step(cuda_lib):
    import torch
    G, D, F, R = 4, 1024, 384, 1152
    routings = [[384, 0, 256, 384], [128, 512, 256, 256], [0, 384, 384, 256]]
    steps = []
    for i, counts in enumerate(routings):
        raw = W.moe_inputs(G, D, F, R, seed=20 + i, dy_seed=30 + i)
        inp = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16) for k, v in raw.items()}
        steps.append((inp, torch.from_numpy(W.offsets_from_counts(counts))))
    got = _pipeline_steps(cuda_lib, steps, G, F, cuda_lib.ACT_SWIGLU, cuda_lib.E4M3, False)
    for i, (inp, offs) in enumerate(steps):
        want = _device_step(cuda_lib, inp, offs, G, F, cuda_lib.ACT_SWIGLU, cuda_lib.E4M3, False)
        A = int(offs[-1])
        for k in ("y", "dx"):
            assert torch.equal(got[i][k][:A], want[k][:A]), (i, k)
        for k in ("dw1", "dw2"):
            assert torch.equal(got[i][k], want[k]), (i, k)


def test_pipeline_dense_gelu_steps_match_device_step(cuda_lib):
    import torch
    M, D, H = 256, 384, 512
    steps = []
    for i in range(3):
        rng = np.random.default_rng(60 + i)
        raw = {"x": W.normal_bf16(rng, (M, D)), "w1": W.normal_bf16(rng, (H, D), std=0.05),
               "w2": W.normal_bf16(rng, (D, H), std=0.05), "dy": W.normal_bf16(rng, (M, D), std=1e-3),
               "b1": W.normal_bf16(rng, (H,), std=0.02), "b2": W.normal_bf16(rng, (D,), std=0.02)}
        inp = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16) for k, v in raw.items()}
        steps.append((inp, None))
    got = _pipeline_steps(cuda_lib, steps, 1, H, cuda_lib.ACT_GELU_TANH, cuda_lib.E2M3, True)
    for i, (inp, _) in enumerate(steps):
        want = _device_step(cuda_lib, inp, None, 1, H, cuda_lib.ACT_GELU_TANH, cuda_lib.E2M3, True)
        for k in want:
            assert torch.equal(got[i][k], want[k]), (i, k)


def test_pipeline_with_resident_weights(cuda_lib):
    """Weights kept on the device (no w1 / w2 / dw1 / dw2 host buffers): each
    step's y and dX come back bitwise equal to the device step's, and the
    last step's weight gradients are left in the device buffers."""
    import torch
    mx = cuda_lib
    G, D, F, R = 4, 1024, 384, 1152
    raw0 = W.moe_inputs(G, D, F, R, seed=40, dy_seed=41)
    to_t = lambda v: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16)
    weights = {k: to_t(raw0[k]) for k in ("w1", "w2")}
    steps = []
    for i, counts in enumerate([[384, 0, 256, 384], [128, 512, 256, 256]]):
        raw = W.moe_inputs(G, D, F, R, seed=42 + i, dy_seed=50 + i)
        inp = {k: to_t(raw[k]) for k in ("x", "dy")}
        inp.update(weights)
        steps.append((inp, torch.from_numpy(W.offsets_from_counts(counts))))
    dev = "cuda"
    dd = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in steps[0][0].items()}
    dd["w1"].copy_(weights["w1"])
    dd["w2"].copy_(weights["w2"])
    dout = {"y": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "dx": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "dw1": torch.empty(weights["w1"].shape, dtype=torch.bfloat16, device=dev),
            "dw2": torch.empty(weights["w2"].shape, dtype=torch.bfloat16, device=dev)}
    doff = torch.empty(G, dtype=torch.int32, device=dev)
    a0 = mx.mlp_args(dd["x"], dd["w1"], dd["w2"], dd["dy"], doff, G, F, dout["y"], dout["dx"], dout["dw1"],
                     dout["dw2"])
    ws = torch.empty(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device=dev)
    a = mx.mlp_args(dd["x"], dd["w1"], dd["w2"], dd["dy"], doff, G, F, dout["y"], dout["dx"], dout["dw1"],
                    dout["dw2"], workspace=ws)
    pipe = mx.MlpPipeline(a)
    results, keep = [], []
    for inp, offs in steps:
        host = {"x": _pinned(inp["x"]), "dy": _pinned(inp["dy"]), "offsets": _pinned(offs)}
        outs = {k: torch.full((R, D), float("nan"), dtype=torch.bfloat16, pin_memory=True) for k in ("y", "dx")}
        host.update(outs)
        pipe.run(host)
        keep.append(host)
        results.append(outs)
    pipe.sync()
    pipe.close()
    assert mx.mx_get_device_status() == "MX_OK"
    for i, (inp, offs) in enumerate(steps):
        want = _device_step(mx, inp, offs, G, F, mx.ACT_SWIGLU, mx.E4M3, False)
        A = int(offs[-1])
        for k in ("y", "dx"):
            assert torch.equal(results[i][k][:A], want[k][:A]), (i, k)
    for k in ("dw1", "dw2"):
        assert torch.equal(dout[k].cpu(), want[k]), k
