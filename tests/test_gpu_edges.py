"""GPU parity at the edges of the standalone calls and of the decode step:
the largest layer shapes of the Llama-3.1-8B and Mixtral-8x7B configurations
(the K = 14336 down projection, the 28672-row gate/up and the 128256-row
lm_head), single-row and single-chunk GEMVs, all-zero weights and inputs,
inputs far from unit size, one-hot columns for every weight type, verification
of the largest draft count, and the decode step's device-side rejection of an
out-of-range position or token (the kernel returns before any copy or barrier
and reports the error; the context stays usable)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import models
import weight_only_quantized_bs_gb300 as gf
from weight_only_quantized_bs_gb300.weights import build_model
from gpu_util import as_f64, bf16_host, rel_err, to_dev, weights, xvec

pytestmark = pytest.mark.gpu

TOL = 1e-2
PER_CHUNK = {oracle.BF16: 8, oracle.INT8: 16, oracle.INT4: 32}
ERR_BAD_POS, ERR_BAD_TOKEN = 7, 8


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert gf.device_error() == 0


def _gemv(dt, W, x, ydt=gf.Y_F32):
    """(GPU y, oracle y) for weights W (bf16 bits) and input x (bf16 bits)."""
    N, K = W.shape
    xd = to_dev(x)
    if dt == oracle.BF16:
        y = gf.gemv_bf16(xd, gf.repack_bf16(to_dev(W)), N, K, ydt)
        ref = oracle.linear(dt, W, None, None, oracle.bf16_to_double(x))
    elif dt == oracle.INT8:
        qp, s = gf.quantize_w8(to_dev(W))
        y = gf.gemv_w8(xd, qp, s, N, K, ydt)
        q, sr = oracle.quant_w8(W)
        ref = oracle.linear(dt, q, sr, None, oracle.bf16_to_double(x))
    else:
        qp = gf.quantize_w4g(to_dev(W))
        y = gf.gemv_w4g(xd, qp, N, K, ydt)
        q, sr, zr = oracle.quant_w4g(W)
        ref = oracle.linear(dt, q, sr, zr, oracle.bf16_to_double(x))
    return as_f64(y), ref


def _scaled_bf16(x, e):
    """x * 2^e, exact for bf16 values well inside the normal range."""
    v = oracle.bf16_to_double(x) * 2.0 ** e
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------ GEMV --
@pytest.mark.slow
@pytest.mark.parametrize("dt", [0, 1, 2])
@pytest.mark.parametrize("N,K", [(6144, 4096), (28672, 4096), (4096, 14336), (128256, 4096)])
def test_gemv_llama31_mixtral_shapes(dt, N, K):
    """Llama-3.1-8B / Mixtral-8x7B layer shapes: GQA qkv, gate/up of ffn 14336,
    the down projection at the largest supported K, the 128256-row lm_head."""
    y, ref = _gemv(dt, weights(N, K, 70 + dt), xvec(K, 71))
    assert rel_err(y, ref) <= 1e-4


@pytest.mark.parametrize("dt", [0, 1, 2])
@pytest.mark.parametrize("N,kc", [(1, 1), (1, 448), (31, 2), (32, 1), (33, 129)])
def test_gemv_single_row_and_chunk(dt, N, kc):
    """One output row, one 16-byte chunk per row, and one row either side of a tile."""
    K = kc * PER_CHUNK[dt]
    y, ref = _gemv(dt, weights(N, K, 72 + dt), xvec(K, 73))
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_gemv_zero_weights_and_zero_input(dt):
    """All-zero weights quantise to s = 0 (and z = 0), q = 0 and give y = 0
    exactly; a zero input gives y = 0 exactly for every weight type."""
    N, K = 45, 1056
    W0 = np.zeros((N, K), np.uint16)
    y, ref = _gemv(dt, W0, xvec(K, 74))
    assert np.all(ref == 0) and np.all(y == 0)
    y, ref = _gemv(dt, weights(N, K, 75), np.zeros(K, np.uint16))
    assert np.all(ref == 0) and np.all(y == 0)


@pytest.mark.parametrize("dt", [0, 1, 2])
@pytest.mark.parametrize("e", [-50, -20, 20, 36])
def test_gemv_input_scale(dt, e):
    """Inputs far from unit size (|x| from about 2^-53 to 2^38): the int4 and
    int8 products stage x multiplied by powers of two up to 2^85, which stays
    finite and keeps the products normal over this whole range."""
    N, K = 100, 4096
    x = _scaled_bf16(xvec(K, 76), e)
    y, ref = _gemv(dt, weights(N, K, 77 + dt), x)
    assert rel_err(y, ref) <= TOL
    assert rel_err(y, ref) <= 1e-4


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_gemv_one_hot_column_every_type(dt):
    """x = e_j returns the dequantised column j exactly (fp32 output), for each
    weight type and at the first, a middle, a chunk-boundary and the last k."""
    N, K = 70, 2048
    W = weights(N, K, 78 + dt)
    if dt == oracle.BF16:
        What = oracle.bf16_to_double(W)
    elif dt == oracle.INT8:
        q, s = oracle.quant_w8(W)
        What = oracle.dequant(dt, q, s)
    else:
        q, s, z = oracle.quant_w4g(W)
        What = oracle.dequant(dt, q, s, z)
    for j in (0, 15, 16, 1031, K - 1):
        x = np.zeros(K, np.uint16)
        x[j] = 0x3F80  # 1.0
        y, _ = _gemv(dt, W, x)
        assert np.allclose(y, What[:, j], rtol=1e-6, atol=1e-7), j


# ----------------------------------------------------------- decode step --
def _step(m, kv, tok, pos, cfg):
    dev = torch.device("cuda")
    t = torch.tensor([tok], dtype=torch.int32, device=dev)
    p = torch.tensor([pos], dtype=torch.int32, device=dev)
    lg = torch.full((cfg["vocab"],), 123.0, dtype=torch.float32, device=dev)
    am = torch.full((1,), -5, dtype=torch.int32, device=dev)
    gf.decode_step(m, kv, t, p, lg, am)
    return int(p.item()), lg.cpu().numpy().astype(np.float64), int(am.item())


def test_decode_rejects_bad_position_and_token():
    cfg = models.config("tiny")
    wc = models.WeightCache(cfg, seed=23)
    m = build_model(cfg, "int8", wc)
    tmax = 16
    kv = gf.KV(m, tmax)
    assert gf.device_error() == 0
    for tok, pos, code in ((3, tmax, ERR_BAD_POS), (3, -1, ERR_BAD_POS), (cfg["vocab"], 0, ERR_BAD_TOKEN),
                           (-1, 0, ERR_BAD_TOKEN)):
        p, lg, am = _step(m, kv, tok, pos, cfg)
        assert gf.device_error() == code, (tok, pos)
        # nothing was written: position, logits and argmax keep their values
        assert p == pos and np.all(lg == 123.0) and am == -5
    # the context is still usable and the cache untouched: a valid step at 0
    # matches the oracle's first step
    p, lg, am = _step(m, kv, 3, 0, cfg)
    assert gf.device_error() == 0 and p == 1
    ref = oracle.OracleModel(cfg, "int8", wc, tmax=tmax).forward([3], 0)[-1]
    assert np.abs(lg - ref).max() <= 2e-2 * ref.std()
    assert am == int(np.argmax(lg))
    kv.close()
    m.close()


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


@pytest.mark.parametrize("dtype", ["int4", "bf16"])
def test_verify_k7_and_a_mismatch_inside(dtype):
    """k = 7 (eight rows, the most one pass takes): all drafts right gives
    n = 7; a wrong draft at index 3 gives n = 3 with the oracle's token there."""
    cfg = models.config("tiny")
    wc = models.WeightCache(cfg, seed=24)
    prompt = list(models.prompt(cfg, 24, 5))
    gen, _ = oracle.OracleModel(cfg, dtype, wc, tmax=64).greedy(prompt, 8)
    m = build_model(cfg, dtype, wc)
    dev = torch.device("cuda")
    k = 7
    bad = list(gen[:k])
    bad[3] = (bad[3] + 1) % cfg["vocab"]
    for drafts in (gen[:k], bad):
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
        got = lg.cpu().numpy().astype(np.float64)
        for i in range(k + 1):
            assert np.abs(got[i] - ref[i]).max() <= 2e-2 * ref[i].std(), i
        assert n_ref == (k if drafts is not bad else 3)
        assert int(n_acc.item()) == n_ref and int(nxt.item()) == nxt_ref == gen[n_ref]
        assert int(pos.item()) == len(prompt) + n_ref
        kv.close()
    m.close()


def test_verify_rejects_rows_past_the_cache():
    """pos + k + 1 > Tmax is refused on the device before any write."""
    cfg = models.config("tiny")
    wc = models.WeightCache(cfg, seed=25)
    m = build_model(cfg, "int8", wc)
    kv = gf.KV(m, 8)
    dev = torch.device("cuda")
    pos = _prefill(m, kv, cfg, [5, 6, 7, 8, 1])       # cache rows 0..3
    toks = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device=dev)
    pos.fill_(5)
    n_acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
    nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
    gf.verify_k(m, kv, toks, 3, pos, n_acc, nxt)
    assert gf.device_error() == ERR_BAD_TOKEN
    assert int(pos.item()) == 5 and int(n_acc.item()) == -1 and int(nxt.item()) == -1
    # the same pass one position earlier fits exactly and runs
    pos.fill_(4)
    gf.verify_k(m, kv, toks, 3, pos, n_acc, nxt)
    assert gf.device_error() == 0 and 0 <= int(n_acc.item()) <= 3
    kv.close()
    m.close()


# ------------------------------------------------------- bounded waits ----
def test_gated_gemv_wait_runs_out_and_context_stays_usable():
    """A grid wait that cannot end: the gated GEMV's CTAs wait for a gate word
    that nothing sets, with a 1 ms limit in place of 2 s.  Every CTA gives up,
    the launch completes, the device error word reads GF_DEVERR_WAIT_GRID and
    nothing was written to y; then the same GEMV behind an open gate, and a
    plain one, match the oracle on the same context."""
    N, K = 4096, 4096  # 128 tiles: 128 CTAs, each with 32 slots behind the gate
    dev = torch.device("cuda")
    W, x = weights(N, K, 90), xvec(K, 91)
    Wp = gf.repack_bf16(to_dev(W))
    xd = to_dev(x)
    ref = oracle.linear(oracle.BF16, W, None, None, oracle.bf16_to_double(x))
    gate = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.full((N,), 7.0, dtype=torch.float32, device=dev)
    assert gf.device_error() == 0
    gf.gemv_bf16_gated(xd, Wp, N, K, gate, 1_000_000, gf.Y_F32, out=y)
    assert gf.device_error() == gf.DEVERR_WAIT_GRID
    assert torch.all(y == 7.0).item()  # nothing past the gate ran
    # the context is usable: the gate opened, then the ungated call
    gate.fill_(1 << 20)
    gf.gemv_bf16_gated(xd, Wp, N, K, gate, 1_000_000_000, gf.Y_F32, out=y)
    assert gf.device_error() == 0
    assert rel_err(as_f64(y), ref) <= 1e-4
    y2 = gf.gemv_bf16(xd, Wp, N, K, gf.Y_F32)
    assert gf.device_error() == 0
    assert rel_err(as_f64(y2), ref) <= 1e-4
