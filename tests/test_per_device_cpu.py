"""The library's one-time launch set-up (dynamic shared-memory opt-in, SM
counts, resident SM pairs) is kept per CUDA device ordinal (csrc/per_device.h),
so a process that drives two GPUs sets each up on both.  Checked on the host:
a small C++ program fills the cache for devices 0 and 1 and counts the fills."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "fp8_scaled_quantization_quantize_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "per_device.h"
using fp8q::PerDevice;
int main() {
    PerDevice<int> cache;
    int fills[fp8q::kMaxDevices] = {};
    auto get = [&](int dev, int& out) {
        return cache.get(dev, out, [&](int& v) { ++fills[dev]; v = 100 + dev; return true; });
    };
    int v = 0;
    // device 0 then device 1 then both again: one fill each, values kept apart
    if (!get(0, v) || v != 100) return 1;
    if (!get(1, v) || v != 101) return 2;
    if (!get(0, v) || v != 100 || !get(1, v) || v != 101) return 3;
    if (fills[0] != 1 || fills[1] != 1) return 4;
    // ordinals outside [0, kMaxDevices) are refused, nothing is filled
    if (get(-1, v) || cache.get(fp8q::kMaxDevices, v, [](int&) { return true; })) return 5;
    // a fill that fails leaves the slot empty, and a later call retries
    PerDevice<bool> attr;
    int tries = 0;
    bool ok = false;
    if (attr.get(3, ok, [&](bool& b) { ++tries; b = false; return false; })) return 6;
    if (!attr.get(3, ok, [&](bool& b) { ++tries; b = true; return true; }) || !ok || tries != 2) return 7;
    if (!attr.get(3, ok, [&](bool& b) { ++tries; return true; }) || tries != 2) return 8;
    // eight host threads on devices 2 and 5: one fill per device
    std::vector<std::thread> th;
    for (int i = 0; i < 8; ++i)
        th.emplace_back([&, i] { int o = 0; get(i % 2 ? 5 : 2, o); });
    for (auto& t : th) t.join();
    if (fills[2] != 1 || fills[5] != 1) return 9;
    std::puts("ok");
    return 0;
}
"""


def test_per_device_cache_is_keyed_by_device():
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.cpp")
        exe = os.path.join(d, "t")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
