"""The benchmark's algorithmic-bytes accounting (the numerator of its roofline
and GB/s figures), checked against an independent count on CPU: per decode
token the streamed weights, every layer's K and V rows 0..pos read once, and
the new row written once."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from synth import models  # noqa: E402


def _count(cfg, weight_bytes, p0, steps):
    """Byte by byte: one bf16 element is 2 bytes; a position holds one K and
    one V vector of head_dim per kv head per layer."""
    total = 0
    per_pos = 0
    for _layer in range(cfg["n_layers"]):
        for _head in range(cfg["n_kv_heads"]):
            per_pos += 2 * cfg["head_dim"] * 2  # K + V, bf16
    for pos in range(p0, p0 + steps):
        total += weight_bytes
        total += per_pos * (pos + 1)  # rows 0..pos read by attention
        total += per_pos              # row pos written
    return total


def test_decode_bytes_matches_an_independent_count():
    for name in ("tiny", "llama2-7b", "llama3.1-8b", "mixtral-8x7b"):
        cfg = models.config(name)
        for p0, steps in ((5, 1), (5, 200), (8195, 32)):
            assert bench.decode_bytes(cfg, 123456789, p0, steps) == _count(cfg, 123456789, p0, steps)


def test_llama2_7b_kv_bytes_per_position():
    # 32 layers x 32 kv heads x 128 dims x (K + V) x 2 bytes = 512 KiB per position
    cfg = models.config("llama2-7b")
    assert bench.decode_bytes(cfg, 0, 0, 1) == 2 * 512 * 1024  # row 0 read, row 0 written
    # Llama-3.1-8B: 8 kv heads, 128 KiB per position
    cfg = models.config("llama3.1-8b")
    assert bench.decode_bytes(cfg, 0, 9, 1) == 11 * 128 * 1024


def test_reference_arm_stages_are_the_oracle_decode():
    """The reference arm's stage stream (one layer, or the final norm and
    lm_head, per step) reproduces the oracle's own token-by-token decode: two
    whole tokens from position 3 after a seeded 3-row context give the
    logits of OracleModel.forward over the same cache."""
    import numpy as np
    import oracle
    from synth import models
    cfg = models.config("tiny")
    st = bench.OracleStream(cfg, "int8", 7, 3, cfg["n_layers"])
    got = []
    for _ in range(2):
        for _ in range(st.n_stages):
            st.stage()
        got.append(st.logits)
    om = oracle.OracleModel(cfg, "int8", models.WeightCache(cfg, seed=7, keep=False), tmax=3 + 64)
    for l in range(cfg["n_layers"]):
        k, v = models.kv_prefill(cfg, 7, l, 3)
        om.K[l][:, :3, :] = oracle.bf16_to_double(k)
        om.V[l][:, :3, :] = oracle.bf16_to_double(v)
    toks = [int(t) for t in models.prompt(cfg, 7, 64)[:2]]
    ref = om.forward(toks, 3)
    assert np.allclose(np.stack(got), ref, rtol=0, atol=1e-12)
