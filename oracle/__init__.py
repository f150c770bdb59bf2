"""The oracle — TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded CPU restatement of the batch-size-1
weight-only-quantised decode step that the gpt-fast pages describe (gpt-fast
README: "Quantization", "Benchmarks", "Speculative sampling"; "Efficiently
implementing the Mixtral 8x7B model with gpt-fast": "Key Features").  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the GPU path: the numeric
primitives are in ``oracle.c`` (built here with gcc), the step structure in
``model.py``.

Parity status of each function (pins are in tests/test_oracle_*.py):
  bf16 conversion, int8 / int4 quantisers, packed layout, linear, attention,
  RMSNorm, RoPE, SwiGLU, decoder layer, MoE FFN, greedy verify: pinned.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

BF16, INT8, INT4 = 0, 1, 2
DTYPES = {"bf16": BF16, "int8": INT8, "int4": INT4}


def build(force=False):
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        vp, lg, i32, dbl = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double
        L.orc_bf16_from_f32.argtypes = [ctypes.c_float]
        L.orc_bf16_from_f32.restype = ctypes.c_uint16
        L.orc_f32_from_bf16.argtypes = [ctypes.c_uint16]
        L.orc_f32_from_bf16.restype = ctypes.c_float
        L.orc_round_bf16.argtypes = [vp, lg]
        L.orc_bf16_to_double.argtypes = [vp, lg, vp]
        L.orc_quant_w8.argtypes = [vp, lg, lg, vp, vp]
        L.orc_quant_w4g.argtypes = [vp, lg, lg, i32, vp, vp, vp]
        L.orc_packed_bytes.argtypes = [i32, lg, lg, i32]
        L.orc_packed_bytes.restype = lg
        L.orc_pack.argtypes = [i32, lg, lg, i32, vp, vp, vp, vp]
        L.orc_unpack.argtypes = [i32, lg, lg, i32, vp, vp, vp, vp]
        L.orc_linear.argtypes = [i32, lg, lg, i32, vp, vp, vp, vp, lg, vp]
        L.orc_attention.argtypes = [i32, i32, i32, lg, vp, vp, vp, vp]
        L.orc_rmsnorm.argtypes = [vp, vp, lg, dbl, vp]
        L.orc_rope.argtypes = [vp, i32, i32, lg, dbl]
        L.orc_swiglu.argtypes = [vp, vp, lg, vp]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16 --
def bf16_from_f32(x):
    """fp32 -> bf16 bit patterns, round to nearest even (element by element)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    L = lib()
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = L.orc_bf16_from_f32(float(flat_in[i]))
    return out


def bf16_to_double(h):
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().orc_bf16_to_double(_p(h), h.size, _p(out))
    return out


def round_bf16(x):
    """Round doubles to bf16 values (double -> fp32 -> bf16, RNE each)."""
    y = np.array(x, dtype=np.float64, copy=True, order="C")
    lib().orc_round_bf16(_p(y), y.size)
    return y


# ------------------------------------------------------------- quantise --
def quant_w8(W):
    """int8 per-output-channel symmetric quantisation of bf16 W [N, K]."""
    W = _c(W, np.uint16)
    N, K = W.shape
    q = np.empty((N, K), dtype=np.int8)
    s = np.empty(N, dtype=np.uint16)
    lib().orc_quant_w8(_p(W), N, K, _p(q), _p(s))
    return q, s


def quant_w4g(W, G=32):
    """int4 grouped (G along K) asymmetric quantisation of bf16 W [N, K]."""
    W = _c(W, np.uint16)
    N, K = W.shape
    assert K % G == 0
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N, K // G), dtype=np.uint16)
    z = np.empty((N, K // G), dtype=np.uint16)
    lib().orc_quant_w4g(_p(W), N, K, G, _p(q), _p(s), _p(z))
    return q, s, z


def group_of(q, s):
    """Group size of int4 codes q [N, K] with per-group scales s [N, K/G]."""
    return q.shape[1] // s.shape[1]


def dequant(dt, q, s=None, z=None):
    """The dequantised weight as fp64 (exact): q*s (int8), q*s+z (int4, the
    group size read off the shapes of q and s)."""
    if dt == BF16:
        return bf16_to_double(q)
    if dt == INT8:
        return q.astype(np.float64) * bf16_to_double(s)[:, None]
    G = group_of(q, s)
    sd = np.repeat(bf16_to_double(s), G, axis=1)
    zd = np.repeat(bf16_to_double(z), G, axis=1)
    return q.astype(np.float64) * sd + zd


# --------------------------------------------------------------- layout --
def packed_bytes(dt, N, K, G=32):
    return int(lib().orc_packed_bytes(dt, N, K, G))


def pack(dt, N, K, src, s=None, z=None, G=32):
    out = np.empty(packed_bytes(dt, N, K, G), dtype=np.uint8)
    src = np.ascontiguousarray(src)
    s = None if s is None else _c(s, np.uint16)
    z = None if z is None else _c(z, np.uint16)
    lib().orc_pack(dt, N, K, G, _p(src), _p(s), _p(z), _p(out))
    return out


def unpack(dt, N, K, packed, G=32):
    packed = _c(packed, np.uint8)
    if dt == BF16:
        dst = np.empty((N, K), dtype=np.uint16)
    elif dt == INT8:
        dst = np.empty((N, K), dtype=np.int8)
    else:
        dst = np.empty((N, K), dtype=np.uint8)
    s = z = None
    if dt == INT4:
        s = np.empty((N, K // G), dtype=np.uint16)
        z = np.empty((N, K // G), dtype=np.uint16)
    lib().orc_unpack(dt, N, K, G, _p(packed), _p(dst), _p(s), _p(z))
    return dst, s, z


# --------------------------------------------------------------- linear --
def linear(dt, w, s, z, X):
    """Y[t] = X[t] . What^T in fp64; X [T, K] (or [K]); w = W / codes [N, K];
    for int4 the group size is K / (columns of s)."""
    w = np.ascontiguousarray(w)
    N, K = w.shape
    X = _c(X, np.float64)
    one = X.ndim == 1
    X2 = X.reshape(-1, K)
    Y = np.empty((X2.shape[0], N), dtype=np.float64)
    s = None if s is None else _c(s, np.uint16)
    z = None if z is None else _c(z, np.uint16)
    G = group_of(w, s) if dt == INT4 else 32
    lib().orc_linear(dt, N, K, G, _p(w), _p(s), _p(z), _p(X2), X2.shape[0], _p(Y))
    return Y[0] if one else Y


def attention(q, Kc, Vc):
    """q [Hq, hd]; Kc, Vc [Hkv, T, hd] (fp64 holding bf16 values) -> [Hq, hd]."""
    q = _c(q, np.float64)
    Kc = _c(Kc, np.float64)
    Vc = _c(Vc, np.float64)
    Hq, hd = q.shape
    Hkv, T, _ = Kc.shape
    out = np.empty((Hq, hd), dtype=np.float64)
    lib().orc_attention(Hq, Hkv, hd, T, _p(q), _p(Kc), _p(Vc), _p(out))
    return out


def rmsnorm(x, g, eps):
    x = _c(x, np.float64)
    g = _c(g, np.uint16)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(g), x.size, float(eps), _p(out))
    return out


def rope(v, nheads, hd, pos, theta):
    v = np.array(v, dtype=np.float64, copy=True, order="C")
    lib().orc_rope(_p(v), nheads, hd, int(pos), float(theta))
    return v


def swiglu(gate, up):
    gate = _c(gate, np.float64)
    up = _c(up, np.float64)
    h = np.empty_like(gate)
    lib().orc_swiglu(_p(gate), _p(up), gate.size, _p(h))
    return h


def argmax(v):
    """Index of the largest value; the lowest index among equal maxima."""
    v = np.asarray(v)
    return int(np.argmax(v))  # numpy returns the first occurrence


from .model import OracleModel  # noqa: E402,F401
