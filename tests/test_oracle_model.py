"""Pins of the oracle's decoder step: an independent brute-force restatement
on a tiny model, zero-weight invariants, MoE routing special cases, and the
speculative-verify rule against plain greedy decoding."""
import math

import numpy as np
import pytest

import oracle
import synth
from synth import models


def f64(h):
    return synth.bf16_to_f32(h).astype(np.float64)


def _bf(x):
    return oracle.round_bf16(x)


def brute_forward(cfg, W, tokens):
    """Plain-loop restatement of the Llama-style step for bf16 weights
    (fp64 activations, bf16 KV cache): written separately from
    oracle/model.py and sharing only the bf16 rounding helper."""
    d, hd, Hq, Hkv = cfg["d"], cfg["head_dim"], cfg["n_heads"], cfg["n_kv_heads"]
    eps, theta = cfg["eps"], cfg["theta"]
    glob = W.glob

    def norm(x, g):
        r = 1.0 / math.sqrt(sum(v * v for v in x) / len(x) + eps)
        return np.array([x[i] * r * g[i] for i in range(len(x))])

    def mat(Wb, x):
        M = f64(Wb)
        return np.array([sum(M[n, k] * x[k] for k in range(M.shape[1])) for n in range(M.shape[0])])

    def rot(v, nh, pos):
        out = v.copy()
        for h in range(nh):
            for i in range(hd // 2):
                a = pos * theta ** (-2.0 * i / hd)
                x0, x1 = v[h * hd + 2 * i], v[h * hd + 2 * i + 1]
                out[h * hd + 2 * i] = x0 * math.cos(a) - x1 * math.sin(a)
                out[h * hd + 2 * i + 1] = x0 * math.sin(a) + x1 * math.cos(a)
        return out

    Kc = [[] for _ in range(cfg["n_layers"])]
    Vc = [[] for _ in range(cfg["n_layers"])]
    logits = []
    for pos, tok in enumerate(tokens):
        x = f64(glob["embed"][tok])
        for l in range(cfg["n_layers"]):
            w = W.layer(l)
            n = norm(x, f64(w["g_attn"]))
            q = rot(mat(w["wq"], n), Hq, pos)
            k = _bf(rot(mat(w["wk"], n), Hkv, pos))   # the KV cache holds bf16
            v = _bf(mat(w["wv"], n))
            Kc[l].append(k)
            Vc[l].append(v)
            att = np.zeros(Hq * hd)
            for h in range(Hq):
                g = h // (Hq // Hkv)
                sc = [sum(q[h * hd + i] * kk[g * hd + i] for i in range(hd)) / math.sqrt(hd) for kk in Kc[l]]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                for i in range(hd):
                    att[h * hd + i] = sum(e[t] * Vc[l][t][g * hd + i] for t in range(len(e))) / sum(e)
            x = x + mat(w["wo"], att)
            mm = norm(x, f64(w["g_ffn"]))
            gt = mat(w["wg"], mm)
            up = mat(w["wu"], mm)
            hh = np.array([gt[i] / (1 + math.exp(-gt[i])) * up[i] for i in range(len(gt))])
            x = x + mat(w["wd"], hh)
        xn = norm(x, f64(glob["g_final"]))
        logits.append(mat(glob["lm_head"], xn))
    return np.array(logits)


def test_decoder_matches_brute_force_tiny():
    cfg = models.config("tiny", d=32, n_heads=2, n_kv_heads=1, head_dim=16, ffn=48, vocab=40,
                        n_layers=2)
    W = models.WeightCache(cfg, seed=3)
    toks = [5, 17, 3]
    ref = brute_forward(cfg, W, toks)
    om = oracle.OracleModel(cfg, "bf16", W, tmax=8)
    got = om.forward(toks, 0)
    assert np.allclose(got, ref, rtol=0, atol=1e-9 * (1 + np.abs(ref).max()))
    # token-by-token decoding equals the layer-major teacher-forced pass
    om2 = oracle.OracleModel(cfg, "bf16", W, tmax=8)
    rows = [om2.forward([t], p)[0] for p, t in enumerate(toks)]
    assert np.allclose(np.stack(rows), got, rtol=0, atol=1e-12)


class _Zeroed:
    def __init__(self, base, names):
        self.base, self.names, self.glob = base, names, base.glob

    def layer(self, l):
        w = dict(self.base.layer(l))
        for n in self.names:
            w[n] = np.zeros_like(w[n])
        return w


@pytest.mark.parametrize("dtype", ["bf16", "int8", "int4"])
def test_zero_output_projections_leave_residual(dtype):
    cfg = models.config("tiny", n_layers=1)
    W = _Zeroed(models.WeightCache(cfg, seed=4), ["wo", "wd"])
    om = oracle.OracleModel(cfg, dtype, W, tmax=4)
    X = f64(W.glob["embed"][[1, 2]])
    out = om.layer_forward(0, X.copy(), 0)
    assert np.array_equal(out, X)


def test_moe_equal_router_logits_pick_first_two_halves():
    cfg = models.config("tiny-moe", n_layers=1)
    base = models.WeightCache(cfg, seed=5)
    W = _Zeroed(base, ["router"])
    om = oracle.OracleModel(cfg, "bf16", W, tmax=4)
    L = om._layer(0)
    m = f64(base.glob["embed"][7])
    (e1, e2), (w1, w2), _ = om.route(L, m)
    assert (e1, e2) == (0, 1) and w1 == 0.5 and w2 == 0.5


def test_moe_zero_expert_leaves_weighted_other():
    cfg = models.config("tiny-moe", n_layers=1)
    base = models.WeightCache(cfg, seed=6)
    om = oracle.OracleModel(cfg, "bf16", base, tmax=4)
    L = om._layer(0)
    m = oracle.round_bf16(f64(base.glob["embed"][9]) * 40)
    (e1, e2), (w1, w2), r = om.route(L, m)
    assert r[e1] >= r[e2] and all(r[e2] >= r[j] for j in range(len(r)) if j not in (e1, e2))
    assert abs(w1 - 1 / (1 + math.exp(r[e2] - r[e1]))) < 1e-15
    # zero the second expert's down projection: output = w1 * y1 (rounded)
    L["experts"][e2]["wd"] = oracle.model._Mat(oracle.BF16, np.zeros_like(base.layer(0)["experts"][e2]["wd"]))
    E = L["experts"][e1]
    y1 = E["wd"](oracle.swiglu(E["wg"](m), E["wu"](m)))
    out = om._ffn_moe(L, m[None, :])[0]
    assert np.array_equal(out, w1 * y1)


@pytest.mark.parametrize("dtype", ["bf16", "int4"])
def test_verify_equals_greedy_decoding(dtype):
    cfg = models.config("tiny")
    W = models.WeightCache(cfg, seed=7)
    prompt = list(models.prompt(cfg, 7, 5))
    ref = oracle.OracleModel(cfg, dtype, W, tmax=32)
    gen, _ = ref.greedy(prompt, 6)
    # target fed the prompt, then asked to verify its own greedy tokens
    om = oracle.OracleModel(cfg, dtype, W, tmax=32)
    om.forward(prompt[:-1], 0)
    n, nxt, lg = om.verify(prompt[-1], gen[:5], len(prompt) - 1)
    assert n == 5 and nxt == gen[5]
    # wrong drafts: the first draft is rejected and the next token is greedy's first
    om2 = oracle.OracleModel(cfg, dtype, W, tmax=32)
    om2.forward(prompt[:-1], 0)
    bad = [(g + 1) % cfg["vocab"] for g in gen[:5]]
    n2, nxt2, _ = om2.verify(prompt[-1], bad, len(prompt) - 1)
    assert n2 == 0 and nxt2 == gen[0]
    # k = 0 is one decoding step
    om3 = oracle.OracleModel(cfg, dtype, W, tmax=32)
    om3.forward(prompt[:-1], 0)
    n3, nxt3, _ = om3.verify(prompt[-1], [], len(prompt) - 1)
    assert n3 == 0 and nxt3 == gen[0]
