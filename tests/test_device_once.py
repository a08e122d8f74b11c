"""The library's one-time set-up per device (csrc/mok_once.h), driven from the host with stub
device ids: a kernel attribute set on one GPU does not carry to another, so the set-up must run once
on every device that launches, exactly once per device under concurrent callers, and again after a
failed attempt.  Plain C++ (g++), no GPU."""
import os
import subprocess

import pytest

from helpers import ROOT

SRC = r'''
#include <cstdio>
#include <thread>
#include <vector>
#include "mok_once.h"

static thread_local int g_dev = 0;
static std::atomic<int> g_calls[4];
static int get_dev(int* d) { *d = g_dev; return 0; }

int main() {
  mok::DeviceOnce once;
  auto setup = [] { g_calls[g_dev].fetch_add(1); return 0; };
  // device 0 twice, then device 1: one set-up each
  g_dev = 0;
  if (once.run(get_dev, setup, 99) || once.run(get_dev, setup, 99)) return 1;
  g_dev = 1;
  if (once.run(get_dev, setup, 99)) return 2;
  if (g_calls[0] != 1 || g_calls[1] != 1) return 3;
  // sixteen threads on devices 2 and 3 at once: still one set-up per device
  std::vector<std::thread> ts;
  for (int i = 0; i < 16; ++i)
    ts.emplace_back([&, i] { g_dev = 2 + (i & 1); for (int k = 0; k < 100; ++k) once.run(get_dev, setup, 99); });
  for (auto& t : ts) t.join();
  if (g_calls[2] != 1 || g_calls[3] != 1) return 4;
  // a failing set-up is reported and retried by the next call
  mok::DeviceOnce again;
  int tries = 0;
  g_dev = 0;
  if (again.run(get_dev, [&] { return ++tries == 1 ? 7 : 0; }, 99) != 7) return 5;
  if (again.run(get_dev, [&] { return ++tries == 1 ? 7 : 0; }, 99) != 0 || tries != 2) return 6;
  if (again.run(get_dev, [&] { return ++tries, 0; }, 99) != 0 || tries != 2) return 7;
  // device ids out of range and a failing device query are errors, not set-ups
  g_dev = 64;
  if (again.run(get_dev, setup, 99) != 99) return 8;
  if (again.run([](int*) { return 5; }, setup, 99) != 5) return 9;
  std::puts("ok");
  return 0;
}
'''


def test_setup_runs_once_per_device(tmp_path):
    if subprocess.run(["which", "g++"], capture_output=True).returncode:
        pytest.skip("g++ not available")
    src = tmp_path / "once.cpp"
    src.write_text(SRC)
    exe = tmp_path / "once"
    inc = os.path.join(ROOT, "mixture_experts_layer_build_gb300", "csrc")
    subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-I", inc, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
