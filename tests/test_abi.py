"""The C-ABI library loads and exports every symbol include/gf.h declares;
host-side argument checks reject bad calls before any launch (no GPU needed);
the library's packed sizes equal the oracle's layout sizes."""
import ctypes
import os
import re

import pytest

import oracle
import weight_only_quantized_bs_gb300 as gf
from weight_only_quantized_bs_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gf.lib()


def declared():
    src = open(os.path.join(ROOT, "include", "gf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gf_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared()
    assert len(names) >= 20
    raw = ctypes.CDLL(gf.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


@pytest.mark.parametrize("dt,N,K", [(0, 4096, 4096), (1, 4096, 11008), (2, 32000, 4096), (2, 45, 1056),
                                    (1, 45, 592), (0, 31, 8), (2, 33, 32), (2, 12288, 4096), (1, 1, 16)])
def test_packed_bytes_match_oracle_layout(L, dt, N, K):
    assert gf.packed_bytes(dt, N, K) == oracle.packed_bytes(dt, N, K)


@pytest.mark.parametrize("N,K,G", [(45, 1056, 32), (45, 1024, 64), (33, 384, 128), (4096, 4096, 128),
                                   (32000, 4096, 64), (1, 128, 128)])
def test_packed_bytes_w4g_match_oracle_layout(L, N, K, G):
    assert gf.packed_bytes(gf.W_INT4G32, N, K, G) == oracle.packed_bytes(2, N, K, G)
    assert L.gf_packed_bytes_w4g(N, K, G) == oracle.packed_bytes(2, N, K, G)


def test_host_checks_reject_before_launch(L):
    vp = ctypes.c_void_p
    assert L.gf_gemv_w4g(None, None, 64, 64, 32, None, 0, None) == 1
    assert L.gf_gemv_w4g(vp(16), vp(16), 64, 64, 48, vp(16), 0, None) == 5        # group size
    assert L.gf_gemv_w4g(vp(16), vp(16), 64, 256, 256, vp(16), 0, None) == 5      # group size
    assert L.gf_gemv_w4g(vp(16), vp(16), 64, 96, 64, vp(16), 0, None) == 5        # G does not divide K
    assert L.gf_gemv_w8(vp(16), vp(16), vp(16), 64, 24, vp(16), 0, None) == 1     # K % 16
    assert L.gf_gemv_bf16(vp(16), vp(16), 64, 64, vp(24), 0, None) == 2           # misaligned y
    assert L.gf_gemv_bf16(vp(16), vp(16), 64, 16384, vp(16), 0, None) == 5        # K > KMAX
    assert L.gf_quantize_w4g(vp(16), 4, 64, 16, vp(16), None) == 5
    assert L.gf_quantize_w4g(vp(16), 4, 96, 64, vp(16), None) == 5
    assert L.gf_unpack_w4g(vp(16), 4, 64, 48, vp(16), vp(16), vp(16), None) == 5
    assert L.gf_kv_reset(None, None) == 1
    assert L.gf_generate(None, None, None, 1, 1, None, None) == 1
    assert L.gf_prefill(None, None, None, 1, None, None, None, None) == 1
    assert L.gf_generate_speculative(None, None, None, None, None, 1, 1, 0, None, None, None) == 1
    ull = ctypes.c_ulonglong
    assert L.gf_gemv_bf16_gated(vp(16), vp(16), 64, 64, vp(16), 0, None, ull(10**6), None) == 1   # no gate
    assert L.gf_gemv_bf16_gated(vp(16), vp(16), 64, 64, vp(16), 0, vp(16), ull(0), None) == 1     # no limit
    assert L.gf_gemv_bf16_gated(vp(16), vp(16), 64, 64, vp(16), 0, vp(18), ull(10**6), None) == 1  # gate align
    assert L.gf_quantize_w8(vp(8), 4, 64, vp(16), vp(16), None) == 2
    assert L.gf_decode_attn(vp(16), vp(16), vp(16), 32, 8, 96, 64, 0, vp(16), vp(16), 1 << 20, None) == 1
    assert L.gf_decode_attn(vp(16), vp(16), vp(16), 32, 8, 128, 64, 64, vp(16), vp(16), 1 << 20, None) == 1
    assert L.gf_copy_ceiling(vp(16), vp(16), 20, None) == 1
    assert L.gf_packed_bytes(2, 64, 48) == -1
    assert L.gf_model_create(None, 0, None, None) == 1
    assert b"gf_model_create" in L.gf_last_error()
