"""GPU parity of the full decode step (gf_decode_step) against the oracle on
small models: teacher-forced on the oracle's own greedy tokens, logits within
2e-2 * std(logits_ref) at every step and an identical argmax wherever the
oracle's top-2 gap exceeds twice that tolerance."""
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


def run_teacher_forced(cfg, dtype, seed, n_prompt, n_gen, tmax):
    wc = models.WeightCache(cfg, seed=seed)
    om = oracle.OracleModel(cfg, dtype, wc, tmax=tmax)
    prompt = list(models.prompt(cfg, seed, n_prompt))
    gen, ref_logits = om.greedy(prompt, n_gen)
    tokens = prompt + gen
    m = build_model(cfg, dtype, wc)
    kv = gf.KV(m, tmax)
    dev = torch.device("cuda")
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    am = torch.empty(1, dtype=torch.int32, device=dev)
    got_logits, got_am = [], []
    for t in tokens:
        tok.fill_(int(t))
        gf.decode_step(m, kv, tok, pos, logits, am)
        got_logits.append(logits.cpu().numpy().astype(np.float64))
        got_am.append(int(am.item()))
    assert int(pos.item()) == len(tokens)
    kv.close()
    m.close()
    return np.stack(got_logits), np.array(got_am), ref_logits


def check(got, got_am, ref):
    skipped = 0
    for i in range(ref.shape[0]):
        tol = 2e-2 * ref[i].std()
        assert np.abs(got[i] - ref[i]).max() <= tol, (i, np.abs(got[i] - ref[i]).max(), tol)
        # the GPU's argmax is the argmax of its own logits
        assert got_am[i] == int(np.argmax(got[i]))
        top2 = np.sort(ref[i])[-2:]
        if top2[1] - top2[0] > 2 * tol:
            assert got_am[i] == int(np.argmax(ref[i])), i
        else:
            skipped += 1
    return skipped


@pytest.mark.parametrize("dtype", ["bf16", "int8", "int4"])
def test_decode_tiny_gqa_200_steps(dtype):
    cfg = models.config("tiny")
    got, am, ref = run_teacher_forced(cfg, dtype, seed=11, n_prompt=5, n_gen=200, tmax=256)
    skipped = check(got, am, ref)
    print("near-tie steps skipped for the argmax check: %d of %d" % (skipped, ref.shape[0]))


@pytest.mark.parametrize("dtype", ["bf16", "int8", "int4"])
def test_decode_small_hd128(dtype):
    cfg = models.config("small")
    got, am, ref = run_teacher_forced(cfg, dtype, seed=12, n_prompt=5, n_gen=12, tmax=64)
    check(got, am, ref)


def test_decode_gqa4_ragged():
    cfg = models.config("tiny", n_heads=8, n_kv_heads=2, d=512, head_dim=64, ffn=736, vocab=1003)
    got, am, ref = run_teacher_forced(cfg, "int4", seed=13, n_prompt=5, n_gen=40, tmax=64)
    check(got, am, ref)


@pytest.mark.parametrize("dtype", ["bf16", "int8", "int4"])
def test_decode_moe_tiny(dtype):
    cfg = models.config("tiny-moe")
    got, am, ref = run_teacher_forced(cfg, dtype, seed=14, n_prompt=5, n_gen=30, tmax=64)
    check(got, am, ref)


def test_decode_moe_mixtral_like():
    """Mixtral structure (8 experts, top-2, GQA 32/8 -> 4, head 128) at small width."""
    cfg = models.config("mixtral-8x7b", d=1024, n_layers=2, n_heads=8, n_kv_heads=2, ffn=1536, vocab=3000)
    got, am, ref = run_teacher_forced(cfg, "int8", seed=15, n_prompt=5, n_gen=10, tmax=32)
    check(got, am, ref)
