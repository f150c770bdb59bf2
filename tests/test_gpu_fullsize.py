"""GPU parity at the full model shapes of the decode workloads, against the
oracle on the same seeded inputs, in the launch configuration the benchmark
times (one persistent launch per decode step on every SM):

* Llama-2-7B-shaped (32 layers), bf16 / int8 / int4-G32: a 6-token
  teacher-forced sequence from position 0, and steps at positions 200..203
  and 2040..2042 after seeded contexts, logits within 2e-2 * std at every
  step and the oracle's argmax (ties within the measured error allowed);
* Llama-3.1-8B-shaped (GQA, vocab 128256): one decode step after a context
  of 128, 1024 or 8192 positions written straight into both KV caches (bf16
  N(0, 1) rows; the workload fixes the context length without a prefill
  run);
* Mixtral-8x7B per-layer shapes (8 experts of ffn 14336, top-2), 2 of the 32
  layers so that the oracle finishes in about a minute: teacher-forced decode
  and a k = 5 speculative verification against the oracle's own verify.

These take minutes (the oracle is plain fp64 C on one core)."""
import numpy as np
import pytest
import torch

import oracle
from synth import models
import weight_only_quantized_bs_gb300 as gf
from weight_only_quantized_bs_gb300.weights import build_model
from gpu_util import check_steps

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert gf.device_error() == 0


class _Raw:
    """A device address where the binding expects a tensor."""

    def __init__(self, p):
        self.p = p

    def data_ptr(self):
        return self.p


def _decode(m, kv, cfg, tokens, pos0):
    dev = torch.device("cuda")
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.full((1,), pos0, dtype=torch.int32, device=dev)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    am = torch.empty(1, dtype=torch.int32, device=dev)
    rows, ams = [], []
    for t in tokens:
        tok.fill_(int(t))
        gf.decode_step(m, kv, tok, pos, lg, am)
        rows.append(lg.cpu().numpy().astype(np.float64))
        ams.append(int(am.item()))
    assert int(pos.item()) == pos0 + len(tokens)
    return np.stack(rows), ams


def check_verify(vgot, vref, toks, n_acc, nxt, n_ref, nxt_ref):
    """Logits rows within tolerance; the device's acceptance is the greedy
    prefix rule applied to its own rows; its argmax of every row that decides
    the acceptance is the oracle's, or a tie within that row's measured logit
    error, and where all of them are the oracle's the acceptance equals the
    oracle's."""
    a = []
    same = True
    for i in range(vref.shape[0]):
        err = float(np.abs(vgot[i] - vref[i]).max())
        tol = 2e-2 * vref[i].std()
        assert err <= tol, (i, err, tol)
        a.append(int(np.argmax(vgot[i])))
        best = int(np.argmax(vref[i]))
        if a[i] != best:
            assert vref[i][a[i]] >= vref[i][best] - 2 * err, i
            if i <= n_ref:
                same = False
    n = 0
    while n < len(toks) - 1 and a[n] == toks[n + 1]:
        n += 1
    assert (n_acc, nxt) == (n, a[n])
    if same:
        assert (n_acc, nxt) == (n_ref, nxt_ref)


def _check(got, ams, ref):
    """At full size the fp32 logits are ~1e-2 from the fp64 oracle's, and a
    32000-way random-init argmax sometimes has a top-2 gap below twice that:
    at most one such tie per run (each within the measured error)."""
    n = check_steps(got, ams, ref)
    print("argmax differs from the oracle's at %d of %d steps" % (n, ref.shape[0]))
    assert n <= 1


@pytest.mark.parametrize("dtype", ["int4", "int8", "bf16"])
def test_llama2_7b_teacher_forced(dtype):
    cfg = models.config("llama2-7b")
    wc = models.WeightCache(cfg, seed=31, keep=False)
    tokens = list(models.prompt(cfg, 31, 6))
    ref = oracle.OracleModel(cfg, dtype, wc, tmax=16, keep=False).forward(tokens, 0)
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, 16)
    got, ams = _decode(m, kv, cfg, tokens, 0)
    kv.close()
    m.close()
    _check(got, ams, ref)


@pytest.mark.slow
@pytest.mark.parametrize("group", [64, 128])
def test_llama2_7b_int4_group_sizes(group):
    """int4 with groups of 64 and 128 along K at the full Llama-2-7B shapes:
    3 teacher-forced steps from position 0."""
    cfg = models.config("llama2-7b", group=group)
    wc = models.WeightCache(cfg, seed=35, keep=False)
    tokens = list(models.prompt(cfg, 35, 3))
    ref = oracle.OracleModel(cfg, "int4", wc, tmax=16, keep=False).forward(tokens, 0)
    m = build_model(cfg, "int4", wc)
    kv = gf.KV(m, 16)
    got, ams = _decode(m, kv, cfg, tokens, 0)
    kv.close()
    m.close()
    _check(got, ams, ref)


@pytest.mark.slow
def test_llama2_7b_prefill_bf16():
    """gf_prefill of a 4-token prompt at the full Llama-2-7B shapes (one
    multi-row pass): the last row's logits and argmax against the oracle's
    forward of the prompt, and the position advanced by 4."""
    cfg = models.config("llama2-7b")
    wc = models.WeightCache(cfg, seed=36, keep=False)
    tokens = [int(t) for t in models.prompt(cfg, 36, 4)]
    ref = oracle.OracleModel(cfg, "bf16", wc, tmax=16, keep=False).forward(tokens, 0)[-1]
    m = build_model(cfg, "bf16", wc)
    kv = gf.KV(m, 16)
    dev = torch.device("cuda")
    toks = torch.tensor(tokens, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    gf.prefill(m, kv, toks, pos, nxt, lg)
    got = lg.cpu().numpy().astype(np.float64)
    kv.close()
    m.close()
    assert int(pos.item()) == 4
    _check(got[None, :], [int(nxt.item())], ref[None, :])


def _write_rows(kv, cfg, tmax, l, k, v, r0, r1):
    """Rows [r0, r1) of layer l's K and V caches (bf16 [Hkv][tmax][hd]) from
    the host arrays k, v ([Hkv][>= r1][hd]), one copy per head."""
    Hkv, hd = cfg["n_kv_heads"], cfg["head_dim"]
    kp, vp = kv.cache_ptrs()
    dev = torch.device("cuda")
    for src, base in ((k, kp), (v, vp)):
        t = torch.from_numpy(np.ascontiguousarray(src[:, r0:r1, :]).view(np.int16)).to(dev)
        for h in range(Hkv):
            off = ((l * Hkv + h) * tmax + r0) * hd * 2
            gf.copy_ceiling(t[h], _Raw(base + off), (r1 - r0) * hd * 2)
    torch.cuda.synchronize()


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["int4", "int8", "bf16"])
def test_llama2_7b_split_kv_positions(dtype):
    """Llama-2-7B at positions the 200-token decode reaches and near the end
    of a 2048-row cache, where attention splits across many CTAs: a seeded
    context of 200 rows in every layer (both caches), 4 teacher-forced steps
    at 200..203, then rows 204..2039 filled the same way and 3 steps at
    2040..2042."""
    cfg = models.config("llama2-7b")
    wc = models.WeightCache(cfg, seed=34, keep=False)
    tmax, L = 2048, cfg["n_layers"]
    om = oracle.OracleModel(cfg, dtype, wc, tmax=tmax, keep=False)
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, tmax)
    draws = []
    for l in range(L):
        k, v = models.kv_prefill(cfg, 34, l, 2040)
        draws.append((k, v))
        om.K[l][:, :200, :] = oracle.bf16_to_double(k[:, :200, :])
        om.V[l][:, :200, :] = oracle.bf16_to_double(v[:, :200, :])
        _write_rows(kv, cfg, tmax, l, k, v, 0, 200)
    toks = list(models.prompt(cfg, 34, 7))
    ref = om.forward(toks[:4], 200)
    got, ams = _decode(m, kv, cfg, toks[:4], 200)
    _check(got, ams, ref)
    for l, (k, v) in enumerate(draws):
        om.K[l][:, 204:2040, :] = oracle.bf16_to_double(k[:, 204:2040, :])
        om.V[l][:, 204:2040, :] = oracle.bf16_to_double(v[:, 204:2040, :])
        _write_rows(kv, cfg, tmax, l, k, v, 204, 2040)
    ref = om.forward(toks[4:], 2040)
    got, ams = _decode(m, kv, cfg, toks[4:], 2040)
    _check(got, ams, ref)
    kv.close()
    m.close()


@pytest.mark.parametrize("dtype,ctx", [("int8", 8192), ("bf16", 8192), ("int8", 128), ("bf16", 1024)])
def test_llama31_8b_long_context(dtype, ctx):
    cfg = models.config("llama3.1-8b")
    wc = models.WeightCache(cfg, seed=32, keep=False)
    tmax = ctx + 8
    Hkv, hd, L = cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"]
    om = oracle.OracleModel(cfg, dtype, wc, tmax=tmax, keep=False)
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, tmax)
    kp, vp = kv.cache_ptrs()
    dev = torch.device("cuda")
    layer_elems = Hkv * tmax * hd
    for l in range(L):
        k, v = models.kv_prefill(cfg, 32, l, ctx)
        om.K[l][:, :ctx, :] = oracle.bf16_to_double(k)
        om.V[l][:, :ctx, :] = oracle.bf16_to_double(v)
        for src, base in ((k, kp), (v, vp)):
            full = np.zeros((Hkv, tmax, hd), dtype=np.uint16)
            full[:, :ctx, :] = src
            t = torch.from_numpy(full.view(np.int16)).to(dev)
            gf.copy_ceiling(t, _Raw(base + l * layer_elems * 2), layer_elems * 2)
    torch.cuda.synchronize()
    token = int(models.prompt(cfg, 32, 1)[0])
    ref = om.forward([token], ctx)
    got, ams = _decode(m, kv, cfg, [token], ctx)
    kv.close()
    m.close()
    _check(got, ams, ref)


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_mixtral_shapes_decode_and_verify(dtype):
    cfg = models.config("mixtral-8x7b", n_layers=2)
    wc = models.WeightCache(cfg, seed=33, keep=True)
    prompt = list(models.prompt(cfg, 33, 5))
    om = oracle.OracleModel(cfg, dtype, wc, tmax=32)
    ref = om.forward(prompt, 0)
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, 32)
    got, ams = _decode(m, kv, cfg, prompt, 0)
    _check(got, ams, ref)
    # k = 5 drafts after the prompt: the oracle's greedy continuation with
    # its third token changed, so that two drafts are accepted
    gen = [int(np.argmax(ref[-1]))]
    om2 = oracle.OracleModel(cfg, dtype, wc, tmax=32)
    om2.forward(prompt, 0)
    for _ in range(4):
        gen.append(int(np.argmax(om2.forward([gen[-1]], len(prompt) + len(gen) - 1)[0])))
    drafts = gen[:5]
    drafts[3] = (drafts[3] + 1) % cfg["vocab"]
    om3 = oracle.OracleModel(cfg, dtype, wc, tmax=32)
    om3.forward(prompt, 0)
    n_ref, nxt_ref, vref = om3.verify(gen[0], drafts[1:] + [gen[4]], len(prompt))
    dev = torch.device("cuda")
    toks = torch.tensor([gen[0]] + drafts[1:] + [gen[4]], dtype=torch.int32, device=dev)
    pos = torch.full((1,), len(prompt), dtype=torch.int32, device=dev)
    n_acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
    nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
    vlg = torch.empty((6, cfg["vocab"]), dtype=torch.float32, device=dev)
    gf.verify_k(m, kv, toks, 5, pos, n_acc, nxt, vlg)
    vgot = vlg.cpu().numpy().astype(np.float64)
    assert n_ref == 2
    check_verify(vgot, vref, toks.cpu().tolist(), int(n_acc.item()), int(nxt.item()), n_ref, nxt_ref)
    assert int(pos.item()) == len(prompt) + int(n_acc.item()) + 1
    kv.close()
    m.close()
