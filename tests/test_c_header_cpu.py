"""include/mx.h as a C header: a C99 program that includes it compiles with
every warning an error, links against the library and gets from the
GPU-free calls (size queries, status strings, host-side rejections) the
same answers as the Python binding.  No GPU: nothing here reaches CUDA."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "mx.h"

int main(void) {
  mx_mlp_args_t a;
  mx_tensor_t t;
  mx_status_t st;
  memset(&a, 0, sizeof a);
  a.act = MX_ACT_SWIGLU;
  a.fmt = MX_E4M3;
  a.G = 128;
  a.R = 262144;
  a.D = 2048;
  a.F = 768;
  printf("abi %d\n", mx_abi_version());
  printf("payload %zu\n", mx_payload_bytes(8192, 7168, MX_E2M3));
  printf("scale %zu\n", mx_scale_bytes(8192, 7168));
  printf("qws %zu\n", mx_quantize_workspace_bytes(8192, 7168, MX_ROWWISE | MX_COLWISE | MX_COLSUM));
  printf("route %lld\n", (long long)mx_moe_route_rows(32768, 8, 128));
  printf("wgws %zu\n", mx_grouped_gemm_wgrad_workspace_bytes(1536, 2048, 262144, 128));
  printf("dgws %zu\n", mx_gemm_dgelu_workspace_bytes(16384, 12288));
  printf("mlpws %zu\n", mx_mlp_workspace_bytes(&a));
  /* rejected by the host validation before any device work: out_row has
     the wrong shape */
  memset(&t, 0, sizeof t);
  t.data = (void *)0x1000;
  t.scale = (uint8_t *)0x2000;
  t.rows = 256;
  t.cols = 128;
  t.fmt = MX_E4M3;
  st = mx_quantize((const void *)0x3000, 1, 256, 256, 256, MX_E4M3, MX_ROWWISE, &t, NULL, NULL, NULL, 0, NULL);
  printf("reject %d %s\n", (int)st, mx_status_string(st));
  printf("names");
  for (int s = MX_OK; s <= MX_ERR_NOT_SUPPORTED; s++) printf(" %s", mx_status_string((mx_status_t)s));
  printf("\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib():
    from mlp_gemms_gb300 import build
    return build.build()


def test_header_compiles_as_c99_and_links(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_SRC)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", libdir, "-lmxgb300", "-Wl,-rpath," + libdir, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = {ln.split(" ", 1)[0]: ln.split(" ", 1)[1] for ln in r.stdout.strip().splitlines()}

    import mlp_gemms_gb300 as mx
    L = mx.load()
    args = mx.MlpArgsStruct()
    args.act, args.fmt, args.G, args.R, args.D, args.F = mx.ACT_SWIGLU, mx.E4M3, 128, 262144, 2048, 768
    want = {
        "abi": str(L.mx_abi_version()),
        "payload": str(L.mx_payload_bytes(8192, 7168, mx.E2M3)),
        "scale": str(L.mx_scale_bytes(8192, 7168)),
        "qws": str(L.mx_quantize_workspace_bytes(8192, 7168, mx.ROWWISE | mx.COLWISE | mx.COLSUM)),
        "route": str(L.mx_moe_route_rows(32768, 8, 128)),
        "wgws": str(L.mx_grouped_gemm_wgrad_workspace_bytes(1536, 2048, 262144, 128)),
        "dgws": str(L.mx_gemm_dgelu_workspace_bytes(16384, 12288)),
        "mlpws": str(L.mx_mlp_workspace_bytes(ctypes.byref(args))),
        "reject": "%d %s" % (mx.STATUS_CODE["MX_ERR_SHAPE"],
                             L.mx_status_string(mx.STATUS_CODE["MX_ERR_SHAPE"]).decode()),
        "names": " ".join(L.mx_status_string(k).decode() for k in sorted(mx.STATUS)),
    }
    assert got == want
    assert int(got["mlpws"]) > 0 and int(got["wgws"]) > 0
