"""Model shapes and seeded random-init weights (bf16 bit patterns).

Shapes are those of the models the gpt-fast benchmark tables name (Llama-2-7B,
Llama-3.1-8B, Mixtral-8x7B); weights are random (no checkpoints exist here).
Distributions: linear weights N(0, 0.02); embedding N(0, 0.02); RMSNorm gains
1 + N(0, 0.02) so that a dropped gain is visible; prompts uniform token ids.
This module only draws numbers: it neither quantises nor computes.
"""
import numpy as np

from . import (TID_EMBED, TID_FINAL_NORM, TID_KV_BASE, TID_LM_HEAD, TID_PROMPT, layer_tid, normal_bf16,
               uniform_int)


def config(name, **over):
    base = {
        # Llama-2-7B-shaped: 32 layers, d 4096, 32 heads x 128, SwiGLU 11008, vocab 32000
        "llama2-7b": dict(d=4096, n_layers=32, n_heads=32, n_kv_heads=32, head_dim=128,
                          ffn=11008, vocab=32000, eps=1e-5, theta=1e4, n_experts=0),
        # Llama-3.1-8B-shaped: GQA 32 q / 8 kv heads, ffn 14336, vocab 128256, theta 5e5
        "llama3.1-8b": dict(d=4096, n_layers=32, n_heads=32, n_kv_heads=8, head_dim=128,
                            ffn=14336, vocab=128256, eps=1e-5, theta=5e5, n_experts=0),
        # Mixtral-8x7B-shaped: 8 experts of ffn 14336, top-2 router, vocab 32000
        "mixtral-8x7b": dict(d=4096, n_layers=32, n_heads=32, n_kv_heads=8, head_dim=128,
                             ffn=14336, vocab=32000, eps=1e-5, theta=1e6, n_experts=8),
        # small shapes that the oracle finishes in seconds; several tiles + ragged tails
        "tiny": dict(d=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64,
                     ffn=352, vocab=1000, eps=1e-5, theta=1e4, n_experts=0),
        "tiny-mha": dict(d=256, n_layers=2, n_heads=4, n_kv_heads=4, head_dim=64,
                         ffn=352, vocab=1000, eps=1e-5, theta=1e4, n_experts=0),
        "tiny-moe": dict(d=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64,
                         ffn=352, vocab=1000, eps=1e-5, theta=1e4, n_experts=4),
        "small": dict(d=1024, n_layers=4, n_heads=8, n_kv_heads=8, head_dim=128,
                      ffn=2816, vocab=5000, eps=1e-5, theta=1e4, n_experts=0),
    }[name]
    base = dict(base)
    base.update(over)
    base["name"] = name
    return base


SIGMA_W = 0.02


def layer_weights(cfg, seed, layer):
    """bf16 weights of one decoder layer (separate q/k/v/gate/up matrices)."""
    d, hd = cfg["d"], cfg["head_dim"]
    Hq, Hkv, F = cfg["n_heads"], cfg["n_kv_heads"], cfg["ffn"]
    t = lambda name, e=0: layer_tid(layer, name, e)  # noqa: E731
    w = {
        "wq": normal_bf16(seed, t("wq"), (Hq * hd, d), SIGMA_W),
        "wk": normal_bf16(seed, t("wk"), (Hkv * hd, d), SIGMA_W),
        "wv": normal_bf16(seed, t("wv"), (Hkv * hd, d), SIGMA_W),
        "wo": normal_bf16(seed, t("wo"), (d, Hq * hd), SIGMA_W),
        "g_attn": normal_bf16(seed, t("g_attn"), (d,), SIGMA_W, mu=1.0),
        "g_ffn": normal_bf16(seed, t("g_ffn"), (d,), SIGMA_W, mu=1.0),
    }
    E = cfg.get("n_experts", 0)
    if E:
        w["router"] = normal_bf16(seed, t("router"), (E, d), SIGMA_W)
        w["experts"] = [{
            "wg": normal_bf16(seed, t("wg", e), (F, d), SIGMA_W),
            "wu": normal_bf16(seed, t("wu", e), (F, d), SIGMA_W),
            "wd": normal_bf16(seed, t("wd", e), (d, F), SIGMA_W),
        } for e in range(E)]
    else:
        w["wg"] = normal_bf16(seed, t("wg"), (F, d), SIGMA_W)
        w["wu"] = normal_bf16(seed, t("wu"), (F, d), SIGMA_W)
        w["wd"] = normal_bf16(seed, t("wd"), (d, F), SIGMA_W)
    return w


def global_weights(cfg, seed):
    d, V = cfg["d"], cfg["vocab"]
    return {
        "embed": normal_bf16(seed, TID_EMBED, (V, d), SIGMA_W),
        "lm_head": normal_bf16(seed, TID_LM_HEAD, (V, d), SIGMA_W),
        "g_final": normal_bf16(seed, TID_FINAL_NORM, (d,), SIGMA_W, mu=1.0),
    }


def kv_prefill(cfg, seed, layer, n_pos):
    """A context of n_pos positions written straight into layer `layer`'s KV
    cache (the long-context decode workloads fix the context length without
    running a prefill): K and V rows bf16 N(0, 1), shape [n_kv_heads, n_pos,
    head_dim] each."""
    shape = (cfg["n_kv_heads"], n_pos, cfg["head_dim"])
    return (normal_bf16(seed, TID_KV_BASE + 2 * layer, shape), normal_bf16(seed, TID_KV_BASE + 2 * layer + 1, shape))


def prompt(cfg, seed, n, tid=TID_PROMPT):
    return uniform_int(seed, tid, n, cfg["vocab"])


class WeightCache:
    """Draws each layer once and keeps it (small models) or re-draws on demand."""

    def __init__(self, cfg, seed, keep=True):
        self.cfg, self.seed, self.keep = cfg, seed, keep
        self._layers = {}
        self.glob = global_weights(cfg, seed)

    def layer(self, l):
        if l in self._layers:
            return self._layers[l]
        w = layer_weights(self.cfg, self.seed, l)
        if self.keep:
            self._layers[l] = w
        return w
