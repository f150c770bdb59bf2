"""Host-side arithmetic of the engine, on CPU: every bulk copy the producer
issues must be 16-byte sized and start 16-byte aligned (an unaligned copy is a
fault, not an error code), and the fused FFN's down slices must cover the
output rows without gaps or overlaps.  A small host program built with nvcc
from the engine's own header enumerates the shapes."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "tests", "_build")

PROGRAM = r"""
#include <cstdio>
#include "gf_internal.cuh"
using namespace gf;

static int bad = 0;
#define CHECK(c, ...) do { if (!(c)) { if (bad < 20) std::printf(__VA_ARGS__); ++bad; } } while (0)

int main() {
  // down slices of a PH_FFN phase: nsl slots of DR rows over d output rows
  for (int dt = 0; dt < 3; ++dt) {
    const int rowb = dt == DT_INT4 ? 12 : dt == DT_INT8 ? 16 : 32;
    for (int d = 16; d <= 16384; d += 16) {
      int nsl, DR;
      ffn_split(dt, d, nsl, DR);
      CHECK(nsl >= 1 && DR % 8 == 0, "dt %d d %d: DR %d\n", dt, d, DR);
      CHECK((long long)DR * rowb <= SLOT_BYTES, "dt %d d %d: slot overflow\n", dt, d);
      CHECK((long long)nsl * DR >= d && (long long)(nsl - 1) * DR < d, "dt %d d %d: slices %d x %d\n", dt, d, nsl, DR);
      for (int k = 0; k < nsl; ++k) {
        const int r0 = k * DR, nr = d - r0 < DR ? d - r0 : DR;
        const long long cb = dt == DT_INT4 ? 8LL * nr : (long long)rowb * nr;
        CHECK(cb % 16 == 0, "dt %d d %d slice %d: code bytes %lld\n", dt, d, k, cb);
        if (dt == DT_INT4) {
          CHECK((4LL * nr) % 16 == 0 && (4LL * r0) % 16 == 0 && (8LL * DR) % 16 == 0,
                "dt %d d %d slice %d: scale copy\n", dt, d, k);
          CHECK((8LL * r0) % 16 == 0, "dt %d d %d slice %d: code offset\n", dt, d, k);
        } else {
          CHECK(((long long)rowb * r0) % 16 == 0, "dt %d d %d slice %d: offset\n", dt, d, k);
        }
      }
    }
  }
  // GEMV slots: every K-block of every tile (ragged last tile, ragged last
  // block) starts on 16 bytes and both its copies are 16-byte sized
  for (int dt = 0; dt < 3; ++dt) {
    const int E = per_chunk(dt);
    for (int N = 1; N <= 100; N += 3) {
      for (int K = E; K <= 2048; K += E * 7) {
        const int C = K / E, nb = (C + KBLK - 1) / KBLK, tiles = (N + TR - 1) / TR;
        long long end = 0;
        for (int t = 0; t < tiles; ++t) {
          const int Rt = N - t * TR < TR ? N - t * TR : TR;
          for (int b = 0; b < nb; ++b) {
            const int Lb = C - b * KBLK < KBLK ? C - b * KBLK : KBLK;
            const long long off = block_offset(dt, C, t, Rt, b);
            CHECK(off % 16 == 0, "dt %d N %d K %d: block offset %lld\n", dt, N, K, off);
            CHECK(off == end, "dt %d N %d K %d: blocks not contiguous\n", dt, N, K);
            end = off + block_bytes(dt, Rt, Lb);
            for (int h = 0; h * HROWS < Rt; ++h) {
              const int r0 = h * HROWS, rh = Rt - r0 < HROWS ? Rt - r0 : HROWS;
              const long long cb = (long long)rh * Lb * 16;
              const long long sb = dt == DT_INT4 ? ((long long)rh * Lb * 4 + 15) / 16 * 16 : 0;
              const long long sz_src = off + (long long)Rt * Lb * 16 + (long long)r0 * Lb * 4;
              CHECK(cb % 16 == 0 && cb <= SLOT_SZ_OFF, "dt %d N %d K %d: code copy %lld\n", dt, N, K, cb);
              CHECK(dt != DT_INT4 || (sz_src % 16 == 0 && sb <= SLOT_BYTES - SLOT_SZ_OFF),
                    "dt %d N %d K %d: scale copy\n", dt, N, K);
            }
          }
        }
        CHECK(end == packed_bytes(dt, N, K), "dt %d N %d K %d: packed size\n", dt, N, K);
      }
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


def test_bulk_copies_aligned_and_down_slices_cover_the_rows():
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
