"""The library's per-device launch-configuration cache (csrc/device_cache.h), compiled into a
small host program with the system C++ compiler: entries for different device ordinals (fake
ones: no GPU is involved) are kept apart, each is computed once, and failed computations are
not remembered."""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_w8a8_quantized_dynamic_gb300", "csrc")

PROGRAM = r"""
#include "device_cache.h"
#include <cstdio>
#include <thread>
#include <vector>
#include <atomic>

int main() {
  fp8k::PerDeviceCache<const void*, int> cache;
  static int kernel_a, kernel_b;
  int calls = 0, v = 0;
  auto compute_for = [&](int value) { return [&, value](int* out) { ++calls; *out = value; return true; }; };
  // device 0 and device 1 hold separate values for the same kernel key
  if (!cache.get(0, &kernel_a, &v, compute_for(10)) || v != 10) return 1;
  if (!cache.get(1, &kernel_a, &v, compute_for(11)) || v != 11) return 2;
  if (!cache.get(0, &kernel_a, &v, compute_for(99)) || v != 10) return 3;  // stored, not recomputed
  if (!cache.get(1, &kernel_a, &v, compute_for(99)) || v != 11) return 4;
  if (!cache.get(1, &kernel_b, &v, compute_for(12)) || v != 12) return 5;
  if (calls != 3 || cache.size() != 3) return 6;
  // a failed computation is not stored: the next call computes again
  int tries = 0;
  auto failing = [&](int* out) { ++tries; *out = 5; return false; };
  if (cache.get(2, &kernel_a, &v, failing)) return 7;
  if (cache.get(2, &kernel_a, &v, failing)) return 8;
  if (tries != 2 || cache.size() != 3) return 9;
  // many host threads on many devices: one computation per (device, key)
  std::atomic<int> computed{0};
  std::vector<std::thread> ts;
  for (int t = 0; t < 16; ++t)
    ts.emplace_back([&, t] {
      int out = 0;
      for (int i = 0; i < 1000; ++i)
        cache.get(100 + (t + i) % 4, &kernel_b, &out, [&](int* o) { computed++; *o = 7; return true; });
    });
  for (auto& th : ts) th.join();
  if (computed.load() != 4) return 10;
  std::puts("ok");
  return 0;
}
"""


def test_per_device_cache_keeps_devices_apart():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "t.cpp"), os.path.join(d, "t")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I" + CSRC, src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
