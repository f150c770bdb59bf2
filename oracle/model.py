"""Decoder step of the oracle, composed from oracle.c's primitives.

TEST INFRASTRUCTURE ONLY.  The step follows the Llama-style transformer that
gpt-fast's model definition serves (gpt-fast README, "Supported models" and
"Generate text"; Mixtral in "Efficiently implementing the Mixtral 8x7B model
with gpt-fast"): embed -> per layer (RMSNorm, q/k/v, RoPE, KV append,
attention, o, residual, RMSNorm, SwiGLU FFN or top-2 MoE, residual) ->
RMSNorm -> lm_head -> fp32 logits -> greedy argmax.

READING of the precision (the pages give none): only the weights are
quantised or kept in bf16, and the KV cache holds bf16 (the decode configs
name it so): k after RoPE and v are rounded to bf16 when they are written to
the cache.  Every other activation -- RMSNorm outputs, q, attention output,
SwiGLU product, linear outputs, the residual stream, logits -- stays at full
precision (fp64 here, fp32 on the GPU).  Speculative
verification (gpt-fast README, "Speculative sampling") accepts the longest
prefix of draft tokens that equals the target's own greedy choices.
"""
import numpy as np

from . import (BF16, INT4, INT8, argmax, attention, bf16_to_double, linear, quant_w4g,
               quant_w8, rmsnorm, rope, round_bf16, swiglu)


class _Mat:
    """One weight matrix as the method stores it: bf16, int8 + s, int4 + s + z
    (group size G along K)."""

    def __init__(self, dt, W, G=32):
        self.dt = dt
        self.N, self.K = W.shape
        if dt == BF16:
            self.w, self.s, self.z = W, None, None
        elif dt == INT8:
            self.w, self.s = quant_w8(W)
            self.z = None
        else:
            self.w, self.s, self.z = quant_w4g(W, G)

    def __call__(self, X):
        return linear(self.dt, self.w, self.s, self.z, X)


class OracleModel:
    """fp64 decoder.  `weights` is a synth.models.WeightCache-like object
    (`.glob`, `.layer(l)`).  Quantised layers are kept when `keep` is set.
    int4 weights use the group size cfg["group"] (32 when absent)."""

    def __init__(self, cfg, dtype, weights, tmax, keep=True):
        self.cfg, self.weights, self.keep = cfg, weights, keep
        self.G = int(cfg.get("group", 32))
        self.dt = {"bf16": BF16, "int8": INT8, "int4": INT4}[dtype] if isinstance(dtype, str) else dtype
        self.tmax = tmax
        c = cfg
        self.K = [np.zeros((c["n_kv_heads"], tmax, c["head_dim"])) for _ in range(c["n_layers"])]
        self.V = [np.zeros((c["n_kv_heads"], tmax, c["head_dim"])) for _ in range(c["n_layers"])]
        self._layers = {}
        self.record = None   # set to a dict to keep the last token's intermediates
        g = weights.glob
        self.embed = g["embed"]
        self.g_final = g["g_final"]
        self.lm_head = _Mat(self.dt, g["lm_head"], self.G)

    def _layer(self, l):
        if l in self._layers:
            return self._layers[l]
        w = self.weights.layer(l)
        G = self.G
        L = {"wq": _Mat(self.dt, w["wq"], G), "wk": _Mat(self.dt, w["wk"], G),
             "wv": _Mat(self.dt, w["wv"], G), "wo": _Mat(self.dt, w["wo"], G),
             "g_attn": w["g_attn"], "g_ffn": w["g_ffn"]}
        if "experts" in w:
            # The router stays bf16: the pages quantise linear weights, and a
            # gate of 8 outputs carries no measurable bytes (READING).
            L["router"] = _Mat(BF16, w["router"])
            L["experts"] = [{k: _Mat(self.dt, e[k], G) for k in ("wg", "wu", "wd")}
                            for e in w["experts"]]
        else:
            for k in ("wg", "wu", "wd"):
                L[k] = _Mat(self.dt, w[k], G)
        if self.keep:
            self._layers[l] = L
        return L

    # -- one layer over T consecutive tokens at positions pos0..pos0+T-1 ------
    def _attn_block(self, l, L, X, pos0):
        c = self.cfg
        T = X.shape[0]
        hd, Hq, Hkv = c["head_dim"], c["n_heads"], c["n_kv_heads"]
        Nrm = np.stack([rmsnorm(X[t], L["g_attn"], c["eps"]) for t in range(T)])
        Q = L["wq"](Nrm)
        Kn = L["wk"](Nrm)
        Vn = round_bf16(L["wv"](Nrm))
        A = np.empty((T, Hq * hd))
        for t in range(T):
            p = pos0 + t
            q = rope(Q[t], Hq, hd, p, c["theta"]).reshape(Hq, hd)
            k = round_bf16(rope(Kn[t], Hkv, hd, p, c["theta"])).reshape(Hkv, hd)
            self.K[l][:, p, :] = k
            self.V[l][:, p, :] = Vn[t].reshape(Hkv, hd)
            A[t] = attention(q, self.K[l][:, :p + 1, :], self.V[l][:, :p + 1, :]).reshape(-1)
        if self.record is not None:
            self.record.update(q=q.reshape(-1), attn=A[-1], k=k.reshape(-1), v=Vn[-1])
        return X + L["wo"](A)

    def _ffn_dense(self, L, M):
        G = L["wg"](M)
        U = L["wu"](M)
        H = np.stack([swiglu(G[t], U[t]) for t in range(M.shape[0])])
        if self.record is not None:
            self.record.update(h=H[-1], gate=G[-1], up=U[-1])
        return L["wd"](H)

    def route(self, L, m):
        """Top-2 of the router logits (lower index first on ties) and the
        softmax over the two chosen logits."""
        r = L["router"](m)
        e1 = argmax(r)
        r2 = r.copy()
        r2[e1] = -np.inf
        e2 = argmax(r2)
        a, b = r[e1], r[e2]
        mx = max(a, b)
        wa, wb = np.exp(a - mx), np.exp(b - mx)
        return (e1, e2), (wa / (wa + wb), wb / (wa + wb)), r

    def _ffn_moe(self, L, M):
        out = np.empty_like(M)
        for t in range(M.shape[0]):
            (e1, e2), (w1, w2), _ = self.route(L, M[t])
            acc = 0.0
            for e, w in ((e1, w1), (e2, w2)):
                E = L["experts"][e]
                y = E["wd"](swiglu(E["wg"](M[t]), E["wu"](M[t])))
                acc = acc + w * y
            out[t] = acc
        return out

    def layer_forward(self, l, X, pos0):
        c = self.cfg
        L = self._layer(l)
        H = self._attn_block(l, L, X, pos0)
        M = np.stack([rmsnorm(H[t], L["g_ffn"], c["eps"]) for t in range(H.shape[0])])
        F = self._ffn_moe(L, M) if "experts" in L else self._ffn_dense(L, M)
        if self.record is not None:
            self.record.update(resid_mid=H[-1], m=M[-1], resid=(H + F)[-1])
        return H + F

    def forward(self, tokens, pos0):
        """Teacher-forced forward of tokens at positions pos0.. (layer-major,
        which equals token-by-token decoding).  Returns fp64 logits [T, V]."""
        tokens = np.asarray(tokens, dtype=np.int64).reshape(-1)
        X = bf16_to_double(self.embed[tokens])
        for l in range(self.cfg["n_layers"]):
            X = self.layer_forward(l, X, pos0)
        Nrm = np.stack([rmsnorm(X[t], self.g_final, self.cfg["eps"]) for t in range(X.shape[0])])
        return self.lm_head(Nrm)

    def greedy(self, prompt, n_new):
        """Prompt fed one token per step, then n_new greedy tokens.  Returns
        (generated tokens, logits of every step)."""
        logits_all, out = [], []
        pos = 0
        tok = None
        for t in list(prompt):
            lg = self.forward([t], pos)[0]
            logits_all.append(lg)
            pos += 1
        tok = argmax(logits_all[-1])
        for _ in range(n_new):
            out.append(tok)
            lg = self.forward([tok], pos)[0]
            logits_all.append(lg)
            pos += 1
            tok = argmax(lg)
        return out, np.stack(logits_all)

    def verify(self, last_token, drafts, pos):
        """Feed [last_token, d1..dk] at positions pos..pos+k; a_i = argmax of
        row i; accept n = the largest n with a_{i-1} == d_i for all i <= n;
        the next token is a_n.  Returns (n, next token, logits [k+1, V])."""
        seq = [int(last_token)] + [int(d) for d in drafts]
        logits = self.forward(seq, pos)
        a = [argmax(row) for row in logits]
        n = 0
        while n < len(drafts) and a[n] == int(drafts[n]):
            n += 1
        return n, a[n], logits
