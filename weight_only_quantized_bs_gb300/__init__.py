"""Python binding of libgf (GB300 / sm_103a): argument marshalling only.

Every step of the decode path runs in the CUDA kernels of ``csrc/``; this
module passes device pointers, sizes and the current CUDA stream through the
C-ABI declared in ``include/gf.h`` and turns status codes into exceptions.
PyTorch supplies device memory and streams.  There is no CPU fallback: if
``libgf.so`` is missing the import of any wrapper raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgf.so")

W_BF16, W_INT8, W_INT4G32 = 0, 1, 2
Y_BF16, Y_F32 = 0, 1
# device error word codes (gf_device_error)
DEVERR_WAIT_GRID = 3
DEVERR_BAD_POS, DEVERR_BAD_TOKEN = 7, 8
TILE_ROWS = 32
KMAX = 14336
DTYPE_NAMES = {"bf16": W_BF16, "int8": W_INT8, "int4": W_INT4G32}

_lib = None


class GfError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise GfError("libgf.so is not built (run __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
        sig = {
            "gf_last_error": ([], ctypes.c_char_p),
            "gf_version": ([], i32),
            "gf_packed_bytes": ([i32, i32, i32], i64),
            "gf_packed_bytes_w4g": ([i32, i32, i32], i64),
            "gf_quantize_w8": ([vp, i32, i32, vp, vp, vp], i32),
            "gf_quantize_w4g": ([vp, i32, i32, i32, vp, vp], i32),
            "gf_repack_bf16": ([vp, i32, i32, vp, vp], i32),
            "gf_unpack_w8": ([vp, i32, i32, vp, vp], i32),
            "gf_unpack_w4g": ([vp, i32, i32, i32, vp, vp, vp, vp], i32),
            "gf_unpack_bf16": ([vp, i32, i32, vp, vp], i32),
            "gf_gemv_bf16": ([vp, vp, i32, i32, vp, i32, vp], i32),
            "gf_gemv_w8": ([vp, vp, vp, i32, i32, vp, i32, vp], i32),
            "gf_gemv_w4g": ([vp, vp, i32, i32, i32, vp, i32, vp], i32),
            "gf_gemv_bf16_gated": ([vp, vp, i32, i32, vp, i32, vp, ctypes.c_ulonglong, vp], i32),
            "gf_attn_workspace_bytes": ([i32, i32, i32], sz),
            "gf_decode_attn": ([vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, sz, vp], i32),
            "gf_decode_attn_noalloc": ([vp, vp, vp, i32, i32, i32, i32, i32, vp, vp], i32),
            "gf_model_create": ([vp, i32, vp, vp], i32),
            "gf_model_destroy": ([vp], i32),
            "gf_model_weight_bytes": ([vp], i64),
            "gf_kv_create": ([vp, i32, vp], i32),
            "gf_kv_destroy": ([vp], i32),
            "gf_kv_reset": ([vp, vp], i32),
            "gf_generate": ([vp, vp, vp, i32, i32, vp, vp], i32),
            "gf_prefill": ([vp, vp, vp, i32, vp, vp, vp, vp], i32),
            "gf_generate_speculative": ([vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp], i32),
            "gf_kv_cache_ptrs": ([vp, vp, vp], i32),
            "gf_decode_step": ([vp, vp, vp, vp, vp, vp, vp], i32),
            "gf_verify_k": ([vp, vp, vp, i32, vp, vp, vp, vp, vp], i32),
            "gf_trace_bytes": ([vp], sz),
            "gf_kv_activation_ptrs": ([vp, vp, vp, vp, vp], i32),
            "gf_decode_step_traced": ([vp, vp, vp, vp, vp, vp, vp, vp], i32),
            "gf_device_error": ([], i32),
            "gf_copy_ceiling": ([vp, vp, sz, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc, what):
    if rc != 0:
        msg = lib().gf_last_error().decode(errors="replace")
        raise GfError("%s failed (status %d): %s" % (what, rc, msg))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def packed_bytes(wdtype, N, K, G=32):
    n = lib().gf_packed_bytes_w4g(N, K, G) if wdtype == W_INT4G32 else lib().gf_packed_bytes(wdtype, N, K)
    if n < 0:
        raise GfError("bad shape for dtype %d: %dx%d (G=%d)" % (wdtype, N, K, G))
    return int(n)


# ------------------------------------------------------------ weights -----
def quantize_w8(W, stream=None):
    N, K = W.shape
    packed = torch.empty(packed_bytes(W_INT8, N, K), dtype=torch.uint8, device=W.device)
    s = torch.empty(N, dtype=torch.bfloat16, device=W.device)
    _check(lib().gf_quantize_w8(_p(W), N, K, _p(packed), _p(s), _s(stream)), "gf_quantize_w8")
    return packed, s


def quantize_w4g(W, G=32, stream=None):
    N, K = W.shape
    packed = torch.empty(packed_bytes(W_INT4G32, N, K, G), dtype=torch.uint8, device=W.device)
    _check(lib().gf_quantize_w4g(_p(W), N, K, G, _p(packed), _s(stream)), "gf_quantize_w4g")
    return packed


def repack_bf16(W, stream=None):
    N, K = W.shape
    packed = torch.empty(packed_bytes(W_BF16, N, K), dtype=torch.uint8, device=W.device)
    _check(lib().gf_repack_bf16(_p(W), N, K, _p(packed), _s(stream)), "gf_repack_bf16")
    return packed


def unpack_w8(packed, N, K, stream=None):
    q = torch.empty((N, K), dtype=torch.int8, device=packed.device)
    _check(lib().gf_unpack_w8(_p(packed), N, K, _p(q), _s(stream)), "gf_unpack_w8")
    return q


def unpack_w4g(packed, N, K, G=32, stream=None):
    dev = packed.device
    q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s = torch.empty((N, K // G), dtype=torch.bfloat16, device=dev)
    z = torch.empty((N, K // G), dtype=torch.bfloat16, device=dev)
    _check(lib().gf_unpack_w4g(_p(packed), N, K, G, _p(q), _p(s), _p(z), _s(stream)), "gf_unpack_w4g")
    return q, s, z


def unpack_bf16(packed, N, K, stream=None):
    W = torch.empty((N, K), dtype=torch.bfloat16, device=packed.device)
    _check(lib().gf_unpack_bf16(_p(packed), N, K, _p(W), _s(stream)), "gf_unpack_bf16")
    return W


# -------------------------------------------------------------- GEMV ------
def _yout(N, ydt, device, out):
    if out is not None:
        return out
    return torch.empty(N, dtype=torch.bfloat16 if ydt == Y_BF16 else torch.float32, device=device)


def gemv_bf16(x, Wp, N, K, ydt=Y_BF16, out=None, stream=None):
    y = _yout(N, ydt, x.device, out)
    _check(lib().gf_gemv_bf16(_p(x), _p(Wp), N, K, _p(y), ydt, _s(stream)), "gf_gemv_bf16")
    return y


def gemv_w8(x, qp, s, N, K, ydt=Y_BF16, out=None, stream=None):
    y = _yout(N, ydt, x.device, out)
    _check(lib().gf_gemv_w8(_p(x), _p(qp), _p(s), N, K, _p(y), ydt, _s(stream)), "gf_gemv_w8")
    return y


def gemv_w4g(x, qp, N, K, ydt=Y_BF16, out=None, G=32, stream=None):
    y = _yout(N, ydt, x.device, out)
    _check(lib().gf_gemv_w4g(_p(x), _p(qp), N, K, G, _p(y), ydt, _s(stream)), "gf_gemv_w4g")
    return y


def gemv_bf16_gated(x, Wp, N, K, gate, wait_ns, ydt=Y_BF16, out=None, stream=None):
    """gf_gemv_bf16 whose CTAs first wait (at most wait_ns) for the int32
    device word `gate` to reach the launch's CTA count."""
    y = _yout(N, ydt, x.device, out)
    _check(lib().gf_gemv_bf16_gated(_p(x), _p(Wp), N, K, _p(y), ydt, _p(gate), int(wait_ns), _s(stream)),
           "gf_gemv_bf16_gated")
    return y


# --------------------------------------------------------- attention ------
def attn_workspace_bytes(Hq, Hkv, hd):
    return int(lib().gf_attn_workspace_bytes(Hq, Hkv, hd))


def decode_attn(q, kcache, vcache, Hq, Hkv, hd, Tmax, pos, out=None, ws=None, stream=None):
    if out is None:
        out = torch.empty(Hq * hd, dtype=torch.bfloat16, device=q.device)
    need = attn_workspace_bytes(Hq, Hkv, hd)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib().gf_decode_attn(_p(q), _p(kcache), _p(vcache), Hq, Hkv, hd, Tmax, pos, _p(out), _p(ws),
                                ws.numel() * ws.element_size(), _s(stream)), "gf_decode_attn")
    return out


def copy_ceiling(src, dst, nbytes, stream=None):
    _check(lib().gf_copy_ceiling(_p(src), _p(dst), nbytes, _s(stream)), "gf_copy_ceiling")


def device_error():
    return int(lib().gf_device_error())


# -------------------------------------------------------- decode step -----
class _Config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("n_experts", ctypes.c_int), ("eps", ctypes.c_float),
                ("theta", ctypes.c_double), ("group_size", ctypes.c_int)]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("g_final", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("wqkv", ctypes.c_void_p), ("wo", ctypes.c_void_p), ("wgu", ctypes.c_void_p),
                ("wd", ctypes.c_void_p), ("g_attn", ctypes.c_void_p), ("g_ffn", ctypes.c_void_p),
                ("router", ctypes.c_void_p)]


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr


class Model:
    """Library-owned quantised weights of a decoder.  `layers` yields, per
    layer, a dict of bf16 device tensors wqkv, wo, wgu (gate/up rows
    interleaved), wd, g_attn, g_ffn -- for a mixture of experts wgu and wd are
    lists (one per expert) and `router` [n_experts][d] is added; `glob` holds
    embed, g_final, lm_head.  cfg["group"] sets the int4 group size (32)."""

    def __init__(self, cfg, wdtype, glob, layers):
        self.cfg = cfg
        self.wdtype = DTYPE_NAMES.get(wdtype, wdtype)
        c = _Config(cfg["d"], cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["ffn"],
                    cfg["vocab"], cfg.get("n_experts", 0), cfg["eps"], cfg["theta"], cfg.get("group", 32))
        keep = []
        arrays = {}
        moe = cfg.get("n_experts", 0) > 0
        for name in ("wqkv", "wo", "wgu", "wd", "g_attn", "g_ffn") + (("router",) if moe else ()):
            if moe and name in ("wgu", "wd"):
                ts = [t for L in layers for t in L[name]]   # layer-major, one per expert
            else:
                ts = [L[name] for L in layers]
            keep.append(ts)
            arrays[name] = _ptr_array(ts)
        cp = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
        w = _Weights(glob["embed"].data_ptr(), glob["g_final"].data_ptr(), glob["lm_head"].data_ptr(),
                     cp(arrays["wqkv"]), cp(arrays["wo"]), cp(arrays["wgu"]), cp(arrays["wd"]),
                     cp(arrays["g_attn"]), cp(arrays["g_ffn"]), cp(arrays["router"]) if moe else None)
        h = ctypes.c_void_p()
        _check(lib().gf_model_create(ctypes.byref(c), self.wdtype, ctypes.byref(w), ctypes.byref(h)),
               "gf_model_create")
        self.h = h

    def weight_bytes(self):
        return int(lib().gf_model_weight_bytes(self.h))

    def close(self):
        if self.h:
            lib().gf_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KV:
    def __init__(self, model, tmax):
        self.model = model
        self.tmax = tmax
        h = ctypes.c_void_p()
        _check(lib().gf_kv_create(model.h, tmax, ctypes.byref(h)), "gf_kv_create")
        self.h = h

    def reset(self, stream=None):
        """Zeroes the cache and step counters (gf_kv_reset); the caller's
        position tensor is theirs to set back to 0."""
        _check(lib().gf_kv_reset(self.h, _s(stream)), "gf_kv_reset")

    def cache_ptrs(self):
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().gf_kv_cache_ptrs(self.h, ctypes.byref(k), ctypes.byref(v)), "gf_kv_cache_ptrs")
        return k.value, v.value

    def activation_ptrs(self):
        q, a, h, r = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().gf_kv_activation_ptrs(self.h, ctypes.byref(q), ctypes.byref(a), ctypes.byref(h),
                                           ctypes.byref(r)), "gf_kv_activation_ptrs")
        return q.value, a.value, h.value, r.value

    def close(self):
        if self.h:
            lib().gf_kv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_step(model, kv, d_token, d_pos, d_logits, d_argmax, stream=None):
    _check(lib().gf_decode_step(model.h, kv.h, _p(d_token), _p(d_pos), _p(d_logits), _p(d_argmax), _s(stream)),
           "gf_decode_step")


def trace_bytes(kv):
    return int(lib().gf_trace_bytes(kv.h))


def decode_step_traced(model, kv, d_token, d_pos, d_logits, d_argmax, d_trace, stream=None):
    """As decode_step, also writing the per-phase, per-CTA trace (int64 tensor
    of trace_bytes(kv) / 8 words) described in include/gf.h."""
    _check(lib().gf_decode_step_traced(model.h, kv.h, _p(d_token), _p(d_pos), _p(d_logits), _p(d_argmax),
                                       _p(d_trace), _s(stream)), "gf_decode_step_traced")


def verify_k(model, kv, d_tokens, k, d_pos, d_n, d_next, d_logits=None, stream=None):
    _check(lib().gf_verify_k(model.h, kv.h, _p(d_tokens), k, _p(d_pos), _p(d_n), _p(d_next), _p(d_logits),
                             _s(stream)), "gf_verify_k")


# -------------------------------------------------------- generation ------
class SpecStats(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_int), ("drafted", ctypes.c_int), ("accepted", ctypes.c_int)]


def _host_ints(seq):
    arr = (ctypes.c_int32 * len(seq))(*[int(t) for t in seq])
    return arr


def prefill(model, kv, tokens, pos, next_token, logits=None, stream=None):
    """gf_prefill: tokens (device int32 [n]) at *pos.. in passes of up to 8
    rows; pos advances by n; next_token <- argmax of the last row."""
    _check(lib().gf_prefill(model.h, kv.h, _p(tokens), int(tokens.numel()), _p(pos), _p(next_token), _p(logits),
                            _s(stream)), "gf_prefill")


def generate(model, kv, prompt, n_new, stream=None):
    """Greedy generation through gf_generate: returns the n_new token ids."""
    hp = _host_ints(prompt)
    out = (ctypes.c_int32 * n_new)()
    _check(lib().gf_generate(model.h, kv.h, hp, len(prompt), n_new, out, _s(stream)), "gf_generate")
    return list(out)


def generate_speculative(target, tkv, draft, dkv, prompt, n_new, k, stream=None):
    """Speculative greedy generation through gf_generate_speculative: returns
    (the n_new token ids, {rounds, drafted, accepted})."""
    hp = _host_ints(prompt)
    out = (ctypes.c_int32 * n_new)()
    st = SpecStats()
    _check(lib().gf_generate_speculative(target.h, tkv.h, draft.h, dkv.h, hp, len(prompt), n_new, k, out,
                                         ctypes.byref(st), _s(stream)), "gf_generate_speculative")
    return list(out), {"rounds": st.rounds, "drafted": st.drafted, "accepted": st.accepted}
