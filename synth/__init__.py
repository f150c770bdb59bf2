"""Seeded synthetic inputs, shared by the GPU harness and the oracle's tests.

Only random draws live here (see synth.c for the generator's definition); the
decode method's arithmetic lives in the package (GPU) and in ``oracle/`` (CPU)
and neither is imported from here.  Tensor ids name each tensor of a model so
that a tensor's values do not depend on which other tensors were drawn.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, src, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, dbl, dbl, vp, i32]
        lib.synth_normal_f32.argtypes = [u64, u64, u64, dbl, dbl, vp, i32]
        lib.synth_uniform_int.argtypes = [u64, u64, u64, ctypes.c_uint32, vp]
        lib.synth_raw.argtypes = [u64, u64, u64]
        lib.synth_raw.restype = u64
        _lib = lib
    return _lib


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def normal_bf16(seed, tid, shape, sigma=1.0, mu=0.0, out=None):
    """bf16 bit patterns (uint16) of mu + sigma*N(0,1), seeded by (seed, tid)."""
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    n = int(np.prod(shape)) if shape else 1
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_bf16(seed, tid, n, float(mu), float(sigma), out.ctypes.data, _threads())
    return out


def normal_f32(seed, tid, shape, sigma=1.0, mu=0.0):
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, out.size, float(mu), float(sigma), out.ctypes.data, _threads())
    return out


def uniform_int(seed, tid, n, range_):
    out = np.empty(int(n), dtype=np.int32)
    _load().synth_uniform_int(seed, tid, int(n), int(range_), out.ctypes.data)
    return out


def raw(seed, tid, j):
    return int(_load().synth_raw(seed, tid, j))


def bf16_to_f32(u16):
    """Exact widening of bf16 bit patterns to float32 (a bit shift)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# Tensor ids of a decoder model: every tensor of layer l gets its own stream.
TID_EMBED, TID_LM_HEAD, TID_FINAL_NORM, TID_PROMPT, TID_X = 1, 2, 3, 4, 5
TID_KV_BASE = 900_000  # pre-filled KV cache rows: TID_KV_BASE + 2 * layer (+1 for V)
_LAYER_BASE = 1000
LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_attn", "g_ffn", "router")


def layer_tid(layer, name, expert=0):
    return _LAYER_BASE + layer * 1000 + LAYER_TENSORS.index(name) * 16 + expert
