"""The per-device kernel-attribute helper (csrc/launch_util.cuh) on the CPU.

A dynamic shared-memory limit belongs to one device's context, so a process that drives
several GPUs must raise it on each.  The helper keeps one bit per device.  This test
compiles the header with g++ against fake `cudaGetDevice` / `cudaFuncSetAttribute`
definitions (no CUDA runtime is linked) and drives it through two devices."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_diffusion_drafter_forward_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

pytestmark = pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                                reason="needs g++ and the CUDA headers")

PROGRAM = r"""
#include <cstdio>
#include <cuda_runtime.h>
#include "launch_util.cuh"

static int g_dev = 0;
static int g_calls[4] = {0, 0, 0, 0};
static int g_fail_next = 0;
extern "C" cudaError_t cudaGetDevice(int* d) { *d = g_dev; return cudaSuccess; }
extern "C" cudaError_t cudaFuncSetAttribute(const void*, cudaFuncAttribute, int) {
  if (g_fail_next) { g_fail_next = 0; return cudaErrorInvalidValue; }
  g_calls[g_dev]++;
  return cudaSuccess;
}
static int g_kernel_stub = 0;
static const void* kern = &g_kernel_stub;  // stands in for a kernel's address

int main() {
  std::atomic<unsigned long long> done{0};
  // device 0 twice: one attribute call
  g_dev = 0; dflash::smem_attr_once(kern, 1000, done); dflash::smem_attr_once(kern, 1000, done);
  // device 1 (a second GPU in the same process): its own call
  g_dev = 1; dflash::smem_attr_once(kern, 1000, done); dflash::smem_attr_once(kern, 1000, done);
  // a failed call leaves the bit clear, so the next call on that device tries again
  g_dev = 2; g_fail_next = 1;
  cudaError_t e = dflash::smem_attr_once(kern, 1000, done);
  dflash::smem_attr_once(kern, 1000, done);
  std::printf("%d %d %d %d %llu\n", g_calls[0], g_calls[1], g_calls[2], (int)e, done.load());
  return 0;
}
"""


def test_attribute_is_raised_once_per_device(tmp_path):
    src = tmp_path / "t.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    cc = subprocess.run(["g++", "-std=c++17", "-I", CUDA_INC, "-I", CSRC, str(src), "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60).stdout.split()
    calls0, calls1, calls2, err, mask = (int(v) for v in out)
    assert (calls0, calls1, calls2) == (1, 1, 1)
    assert err != 0            # the failure was reported to the caller
    assert mask == 0b111       # devices 0, 1 and (after its retry) 2


def test_every_launcher_uses_the_per_device_helper():
    """No kernel launcher keeps a once-per-process attribute flag."""
    for name in os.listdir(CSRC):
        if not name.endswith(".cu"):
            continue
        text = open(os.path.join(CSRC, name)).read()
        if "cudaFuncAttributeMaxDynamicSharedMemorySize" in text:
            pytest.fail(f"{name} sets the shared-memory attribute directly")
