"""Host-side arithmetic of the engine, on CPU: every weight slot is one
16-byte-sized bulk copy that fits its shared-memory ring entry, the
layout's address functions place every code byte and scale word of a matrix
in a distinct byte of the packed buffer, every bulk copy of the fused FFN's
down pieces starts on a 16-byte boundary and is 16-byte sized (a misaligned
copy is a fault, not an error code), and the down pieces cover the output
rows without gaps or overlaps.  A small host
program built with nvcc from the engine's own header enumerates the shapes."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "tests", "_build")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "gf_internal.cuh"
using namespace gf;

static int bad = 0;
#define CHECK(c, ...) do { if (!(c)) { if (bad < 20) std::printf(__VA_ARGS__); ++bad; } } while (0)

int main() {
  // GEMV slots: one bulk copy per slot (16-byte sized), fitting a ring
  // entry; code_addr / sz_addr place every code byte and scale word of a
  // matrix in a distinct byte inside the packed buffer; the staged input with
  // its zero tail fits the x area
  const int groups[3] = {32, 64, 128};
  for (int dt = 0; dt < 3; ++dt) {
    for (int gi = 0; gi < (dt == DT_INT4 ? 3 : 1); ++gi) {
      const int G = dt == DT_INT4 ? groups[gi] : 32;
      CHECK(slot_bytes(dt, G) <= SLOT_BYTES && slot_bytes(dt, G) % 128 == 0,
            "dt %d G %d: slot %d bytes\n", dt, G, slot_bytes(dt, G));
      const int step = dt == DT_INT4 ? G : per_chunk(dt);
      for (int K = step; K <= KMAX; K += step * ((K / step) % 13 + 1)) {
        CHECK(round_up(K, slot_k(dt)) <= KMAX, "dt %d K %d: staged tail\n", dt, K);
        const long long rowb = dt == DT_BF16 ? 2LL * K : dt == DT_INT8 ? K : K / 2;
        CHECK(k_slots(dt, K) * 256LL >= rowb && (k_slots(dt, K) - 1) * 256LL < rowb, "dt %d K %d: K-slots\n", dt, K);
      }
      for (int N = 1; N <= 70; N += 23) {
        const int K = dt == DT_INT4 ? 3 * G + 512 : 3 * per_chunk(dt) + slot_k(dt);
        const long long rowb = dt == DT_BF16 ? 2LL * K : dt == DT_INT8 ? K : K / 2;
        const long long pb = packed_bytes(dt, N, K, G);
        std::vector<unsigned char> used(pb, 0);
        for (int n = 0; n < N; ++n)
          for (long long j = 0; j < rowb; ++j) {
            const long long a = code_addr(dt, K, G, n, j);
            CHECK(a >= 0 && a < pb && !used[a], "dt %d N %d K %d: code byte %d %lld -> %lld\n", dt, N, K, n, j, a);
            if (a >= 0 && a < pb) used[a] = 1;
          }
        if (dt == DT_INT4)
          for (int n = 0; n < N; ++n)
            for (int g = 0; g < K / G; ++g) {
              const long long a = sz_addr(K, G, n, g);
              CHECK(a >= 0 && a + 4 <= pb && a % 4 == 0, "G %d N %d: scale word %d %d\n", G, N, n, g);
              for (int i = 0; i < 4 && a >= 0 && a + i < pb; ++i) {
                CHECK(!used[a + i], "G %d N %d: scale word %d %d overlaps\n", G, N, n, g);
                used[a + i] = 1;
              }
            }
      }
    }
  }
  // down pieces of a PH_FFN phase: the NCW warps' pieces cover the d output
  // rows exactly once; every copy is 16-byte sized and aligned; a piece fits
  // its slot; the phase's shared buffers fit beside the staged input
  for (int dt = 0; dt < 3; ++dt) {
    for (int d = 32; d <= 7040; d += 32) {
      const FfnSplit fs = ffn_split(dt, d);
      CHECK(fs.RW % 32 == 0 && fs.PR % 32 == 0 && fs.P >= 1, "dt %d d %d: split\n", dt, d);
      CHECK((long long)fs.PR * ffn_row_bytes(dt) <= SLOT_BYTES, "dt %d d %d: piece overflow\n", dt, d);
      std::vector<int> seen(d, 0);
      for (int w = 0; w < NCW; ++w)
        for (int k = 0; k < fs.P; ++k) {
          int r0, r1;
          ffn_piece(fs, d, w, k, r0, r1);
          if (r0 >= r1) continue;
          const long long nr = r1 - r0;
          CHECK(nr <= fs.PR, "dt %d d %d: piece rows\n", dt, d);
          for (int r = r0; r < r1; ++r) ++seen[r];
          if (dt == DT_INT4) {
            CHECK((8LL * r0) % 16 == 0 && (8LL * nr) % 16 == 0 && (4LL * r0) % 16 == 0 && (4LL * nr) % 16 == 0 &&
                  (8LL * fs.PR) % 16 == 0, "dt %d d %d w %d k %d: int4 copies\n", dt, d, w, k);
          } else {
            CHECK((16LL * r0) % 16 == 0 && (16LL * fs.PR) % 16 == 0, "dt %d d %d: copies\n", dt, d);
          }
        }
      for (int r = 0; r < d; ++r) CHECK(seen[r] == 1, "dt %d d %d: row %d covered %d times\n", dt, d, r, seen[r]);
    }
  }
  if (bad) {
    std::printf("%d violations\n", bad);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
"""


def test_slots_fit_and_down_pieces_cover_the_rows():
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if not nvcc:
        pytest.skip("nvcc not available")
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(BUILD, "host_layout.cu")
    exe = os.path.join(BUILD, "host_layout")
    with open(src, "w") as f:
        f.write(PROGRAM)
    csrc = os.path.join(ROOT, "weight_only_quantized_bs_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", csrc, "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout
