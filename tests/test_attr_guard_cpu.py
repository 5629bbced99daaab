"""The kernel launch-attribute guard (mlp_gemms_gb300/csrc/attr_guard.h)
keys on the device: cudaFuncSetAttribute acts on the current device only,
so a process that drives several GPUs must set it once per device and per
kernel.  Host logic, compiled here with g++ against a stand-in CUDA runtime
header that records the calls."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mlp_gemms_gb300", "csrc")

FAKE_RUNTIME = r'''
#pragma once
typedef int cudaError_t;
enum { cudaSuccess = 0, cudaErrorInvalidDevice = 101 };
enum cudaFuncAttribute { cudaFuncAttributeMaxDynamicSharedMemorySize = 8 };
inline int g_dev = 0;
inline bool g_fail_get = false;
inline int g_calls[80][2] = {};
void k_a();
void k_b();
inline cudaError_t cudaGetDevice(int* d) { if (g_fail_get) return cudaErrorInvalidDevice; *d = g_dev; return cudaSuccess; }
template <class T> cudaError_t cudaFuncSetAttribute(T k, cudaFuncAttribute, int) {
  g_calls[g_dev][k == &k_a ? 0 : 1]++;
  return cudaSuccess;
}
'''

MAIN = r'''
#include "attr_guard.h"
#include <cstdio>
#include <initializer_list>
void k_a() {}
void k_b() {}
int main() {
  for (int rep = 0; rep < 3; rep++) {
    for (int d : {0, 1, 5, 70}) {
      g_dev = d;
      if (mx::ensure_smem_attr<&k_a>(1000) != cudaSuccess) return 1;
      if (mx::ensure_smem_attr<&k_b>(1000) != cudaSuccess) return 1;
    }
  }
  g_fail_get = true;
  if (mx::ensure_smem_attr<&k_a>(1000) == cudaSuccess) return 2;   // the device query's error is returned
  std::printf("%d %d %d %d %d %d %d %d\n", g_calls[0][0], g_calls[0][1], g_calls[1][0], g_calls[1][1],
              g_calls[5][0], g_calls[5][1], g_calls[70][0], g_calls[70][1]);
  return 0;
}
'''


def test_attribute_set_once_per_device_and_kernel(tmp_path):
    fake = tmp_path / "fake"
    fake.mkdir()
    (fake / "cuda_runtime.h").write_text(FAKE_RUNTIME)
    src = tmp_path / "main.cpp"
    src.write_text(MAIN)
    exe = tmp_path / "guard"
    r = subprocess.run(["g++", "-std=c++17", "-I", str(fake), "-I", CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.fail(r.stderr)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.returncode
    # devices 0, 1, 5: once per kernel; ordinal 70 (past the mask): every call
    assert out.stdout.split() == ["1", "1", "1", "1", "1", "1", "3", "3"]
