"""The tag arithmetic of the fused decode kernel's hand-off words, checked on the CPU.

The kernel and this test compile the same header (bit_expert_layer_gb300/csrc/
decode_tag.h) -- here with the host C++ compiler.  Over one whole epoch period the tags
must be nonzero (a word never written is zero), distinct for distinct (epoch, layer)
pairs (they increase strictly in epoch-major order), free of 32-bit overflow, and the
epoch must wrap to 0 after the period's last launch.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_expert_layer_gb300", "csrc")

PROG = r"""
#include <cstdint>
#include <cstdio>
#include "decode_tag.h"
using namespace moe;
int main() {
  const int L = 1 << DEC_TAG_LAYER_BITS;
  uint64_t prev = 0;
  for (uint64_t e = 0; e < DEC_EPOCH_PERIOD; ++e) {
    const uint64_t lo = dec_tag(static_cast<uint32_t>(e), 0), hi = dec_tag(static_cast<uint32_t>(e), L - 1);
    const uint64_t lo_exact = (e + 1) * L, hi_exact = (e + 1) * L + L - 1;
    if (lo != lo_exact || hi != hi_exact) { printf("overflow at epoch %llu\n", (unsigned long long)e); return 1; }
    if (lo == 0 || lo <= prev) { printf("not increasing at epoch %llu\n", (unsigned long long)e); return 2; }
    prev = hi;
    const uint32_t n = dec_next_epoch(static_cast<uint32_t>(e));
    if (e + 1 < DEC_EPOCH_PERIOD ? n != e + 1 : n != 0) { printf("next epoch wrong at %llu\n", (unsigned long long)e); return 3; }
  }
  printf("ok %u %llu\n", DEC_EPOCH_PERIOD, (unsigned long long)prev);
  return 0;
}
"""


def test_decode_tag_arithmetic(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "tag.cpp"
    src.write_text(PROG)
    exe = tmp_path / "tag"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    period, last = r.stdout.split()[1:]
    assert int(period) == 2 ** 26 - 1
    assert int(last) == 2 ** 32 - 1           # the last tag of a period is the largest 32-bit value
