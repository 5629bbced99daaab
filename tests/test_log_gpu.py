"""MX_LOG=1: the library prints each launch configuration once per process
(kernel, epilogue, tile width, shapes, grid), however often it launches."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SNIPPET = r'''
import torch, mlp_gemms_gb300 as mx
mx.load()
x = torch.randn((256, 512), device="cuda").to(torch.bfloat16)
w = torch.randn((256, 512), device="cuda").to(torch.bfloat16)
offs = torch.tensor([256], dtype=torch.int32, device="cuda")
for _ in range(3):
    xr, _, _ = mx.mx_quantize(x, mx.E4M3, True, False)
    wr, _, _ = mx.mx_quantize(w, mx.E4M3, True, False)
    mx.mx_grouped_gemm(xr, wr, 1, offs)
w2 = torch.randn((512, 512), device="cuda").to(torch.bfloat16)
w2r, _, _ = mx.mx_quantize(w2, mx.E4M3, True, False)
mx.mx_grouped_gemm(xr, w2r, 1, offs)
torch.cuda.synchronize()
assert mx.mx_get_device_status() == "MX_OK"
'''


def test_mx_log_prints_each_configuration_once(cuda_lib):
    env = dict(os.environ, MX_LOG="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", SNIPPET], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("mx: ")]
    gemm = [l for l in lines if l.startswith("mx: gemm ")]
    quant = [l for l in lines if l.startswith("mx: quantize ")]
    assert len(lines) == len(set(lines)), lines                  # nothing twice
    assert len(gemm) == 2, gemm                                  # N = 256 and N = 512
    assert any("N=256" in l for l in gemm) and any("N=512" in l for l in gemm)
    assert len(quant) == 2, quant                                # [256, 512] and [512, 512]
    env.pop("MX_LOG")
    r = subprocess.run([sys.executable, "-c", SNIPPET], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and not any(l.startswith("mx: ") for l in r.stderr.splitlines())
