"""GPU parity of speculative verification (gf_verify_k) against the oracle:
k+1 rows [last token, drafts] through every layer in one weight pass; the
logits of every row match the oracle's teacher-forced forward, the accepted
count and next token follow the greedy-prefix rule, the position advances by
n + 1, and decoding continues from the KV rows the pass wrote."""
import numpy as np
import pytest
import torch

import oracle
from synth import models
import weight_only_quantized_bs_gb300 as gf
from weight_only_quantized_bs_gb300.weights import build_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert gf.device_error() == 0


def _prefill(m, kv, cfg, prompt):
    dev = torch.device("cuda")
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    am = torch.empty(1, dtype=torch.int32, device=dev)
    for t in prompt[:-1]:
        tok.fill_(int(t))
        gf.decode_step(m, kv, tok, pos, lg, am)
    return pos


def _check_rows(got, ref):
    for i in range(ref.shape[0]):
        tol = 2e-2 * ref[i].std()
        assert np.abs(got[i] - ref[i]).max() <= tol, (i, np.abs(got[i] - ref[i]).max(), tol)


@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("tiny", "int4"), ("small", "int8"), ("tiny-moe", "int8"),
                                        ("tiny-moe", "int4")])
def test_verify_matches_oracle(name, dtype):
    cfg = models.config(name)
    wc = models.WeightCache(cfg, seed=21)
    prompt = list(models.prompt(cfg, 21, 5))
    gen, _ = oracle.OracleModel(cfg, dtype, wc, tmax=64).greedy(prompt, 7)
    m = build_model(cfg, dtype, wc)
    dev = torch.device("cuda")
    k = 5
    for drafts, expect_n in ((gen[:k], k), ([(g + 1) % cfg["vocab"] for g in gen[:k]], 0)):
        kv = gf.KV(m, 64)
        pos = _prefill(m, kv, cfg, prompt)
        toks = torch.tensor([prompt[-1]] + list(drafts), dtype=torch.int32, device=dev)
        n_acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
        nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
        lg = torch.empty((k + 1, cfg["vocab"]), dtype=torch.float32, device=dev)
        gf.verify_k(m, kv, toks, k, pos, n_acc, nxt, lg)
        om = oracle.OracleModel(cfg, dtype, wc, tmax=64)
        om.forward(prompt[:-1], 0)
        n_ref, nxt_ref, ref = om.verify(prompt[-1], drafts, len(prompt) - 1)
        _check_rows(lg.cpu().numpy().astype(np.float64), ref)
        assert n_ref == expect_n
        assert int(n_acc.item()) == n_ref and int(nxt.item()) == nxt_ref == gen[n_ref]
        assert int(pos.item()) == len(prompt) + n_ref
        # decoding continues from the cache rows the pass wrote (rows past the
        # accepted ones are overwritten)
        tok = torch.tensor([int(nxt.item())], dtype=torch.int32, device=dev)
        lg1 = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
        am = torch.empty(1, dtype=torch.int32, device=dev)
        gf.decode_step(m, kv, tok, pos, lg1, am)
        om2 = oracle.OracleModel(cfg, dtype, wc, tmax=64)
        seq = prompt + gen[:n_ref + 1]
        ref1 = om2.forward(seq, 0)[-1]
        _check_rows(lg1.cpu().numpy().astype(np.float64)[None], ref1[None])
        kv.close()
    m.close()


def test_verify_k0_is_a_decode_step():
    cfg = models.config("tiny")
    wc = models.WeightCache(cfg, seed=22)
    prompt = list(models.prompt(cfg, 22, 5))
    gen, _ = oracle.OracleModel(cfg, "int4", wc, tmax=32).greedy(prompt, 1)
    m = build_model(cfg, "int4", wc)
    kv = gf.KV(m, 32)
    pos = _prefill(m, kv, cfg, prompt)
    dev = torch.device("cuda")
    toks = torch.tensor([prompt[-1]], dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.zeros(1, dtype=torch.int32, device=dev)
    gf.verify_k(m, kv, toks, 0, pos, n_acc, nxt)
    assert int(n_acc.item()) == 0 and int(nxt.item()) == gen[0] and int(pos.item()) == len(prompt)
    kv.close()
    m.close()


@pytest.mark.parametrize("name,target,draft,k", [("tiny", "bf16", "int4", 4), ("small", "int8", "int4", 3),
                                                 ("tiny", "int8", "int8", 7), ("tiny-moe", "int8", "int4", 3)])
def test_speculative_generation_equals_greedy(name, target, draft, k):
    """gf_generate_speculative (a draft copy of the same seeded model in
    another weight type proposes k tokens, the target verifies) emits exactly
    the oracle's plain greedy decode of the target over 40 tokens, and so
    does gf_generate on the target; with the draft equal to the target's own
    weights almost every draft is accepted."""
    cfg = models.config(name)
    wc = models.WeightCache(cfg, seed=24)
    prompt = [int(t) for t in models.prompt(cfg, 24, 5)]
    n_new = 40
    ref, _ = oracle.OracleModel(cfg, target, wc, tmax=64).greedy(prompt, n_new)
    tm = build_model(cfg, target, wc)
    dm = build_model(cfg, draft, wc)
    tkv, dkv = gf.KV(tm, 64), gf.KV(dm, 64)
    plain = gf.generate(tm, tkv, prompt, n_new)
    assert plain == [int(t) for t in ref]
    spec, st = gf.generate_speculative(tm, tkv, dm, dkv, prompt, n_new, k)
    assert spec == [int(t) for t in ref]
    assert st["drafted"] == st["rounds"] * k and 0 <= st["accepted"] <= st["drafted"]
    # every round emits accepted + 1 tokens (the first also the prompt's next)
    assert st["accepted"] + st["rounds"] + 1 >= n_new
    if draft == target:
        assert st["accepted"] >= 0.9 * st["drafted"]
    for h in (tkv, dkv):
        h.close()
    tm.close()
    dm.close()
    assert gf.device_error() == 0


@pytest.mark.parametrize("name,dtype,n", [("tiny", "int8", 5), ("tiny", "int4", 13), ("small", "bf16", 8),
                                          ("tiny-moe", "int8", 11)])
def test_prefill_matches_oracle_and_continues(name, dtype, n):
    """gf_prefill feeds an n-token prompt in passes of up to 8 rows (one
    weight stream each): the last row's logits match the oracle's forward of
    the prompt, its argmax is the next token, the position advances by n,
    and decoding from the rows it wrote matches the oracle's continuation."""
    cfg = models.config(name)
    wc = models.WeightCache(cfg, seed=25)
    prompt = [int(t) for t in models.prompt(cfg, 25, n)]
    om = oracle.OracleModel(cfg, dtype, wc, tmax=64)
    ref = om.forward(prompt, 0)
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, 64)
    dev = torch.device("cuda")
    toks = torch.tensor(prompt, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    gf.prefill(m, kv, toks, pos, nxt, lg)
    assert int(pos.item()) == n
    got = lg.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref[-1]).max() <= 2e-2 * ref[-1].std()
    assert int(nxt.item()) == int(np.argmax(got))
    # three decode steps on the prefilled cache against the oracle's
    t = int(np.argmax(ref[-1]))
    am = torch.empty(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    for step in range(3):
        rref = om.forward([t], n + step)[0]
        tok.fill_(t)
        gf.decode_step(m, kv, tok, pos, lg, am)
        g = lg.cpu().numpy().astype(np.float64)
        assert np.abs(g - rref).max() <= 2e-2 * rref.std(), step
        t = int(np.argmax(rref))
    kv.close()
    m.close()
    assert gf.device_error() == 0
