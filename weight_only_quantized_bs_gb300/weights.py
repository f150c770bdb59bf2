"""Host bf16 weights (uint16 bit patterns, one array per matrix) -> the fused
device tensors gf_model_create reads: wqkv = rows of Wq, Wk, Wv stacked;
wgu = gate and up rows interleaved (row 2j = gate j, row 2j+1 = up j).
Row placement only; no arithmetic."""
import numpy as np
import torch


def to_dev(a, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device, non_blocking=False).view(torch.bfloat16)


def _interleave(wg, wu):
    wgu = np.empty((2 * wg.shape[0], wg.shape[1]), dtype=np.uint16)
    wgu[0::2] = wg
    wgu[1::2] = wu
    return wgu


def fuse_layer(w, device="cuda"):
    out = {
        "wqkv": to_dev(np.concatenate([w["wq"], w["wk"], w["wv"]], axis=0), device),
        "wo": to_dev(w["wo"], device),
        "g_attn": to_dev(w["g_attn"], device),
        "g_ffn": to_dev(w["g_ffn"], device),
    }
    if "experts" in w:
        out["wgu"] = [to_dev(_interleave(e["wg"], e["wu"]), device) for e in w["experts"]]
        out["wd"] = [to_dev(e["wd"], device) for e in w["experts"]]
        out["router"] = to_dev(w["router"], device)
    else:
        out["wgu"] = to_dev(_interleave(w["wg"], w["wu"]), device)
        out["wd"] = to_dev(w["wd"], device)
    return out


def device_globals(g, device="cuda"):
    return {k: to_dev(g[k], device) for k in ("embed", "g_final", "lm_head")}


def build_model(cfg, wdtype, weights, device="cuda"):
    """Quantises a synthetic model layer by layer (each layer's bf16 copy is
    released once its quantised form exists)."""
    from . import Model
    glob = device_globals(weights.glob, device)
    layers = [fuse_layer(weights.layer(l), device) for l in range(cfg["n_layers"])]
    m = Model(cfg, wdtype, glob, layers)
    del layers, glob
    return m
