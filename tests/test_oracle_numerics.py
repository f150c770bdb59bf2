"""Pins of the oracle's primitives against facts fixed outside the oracle:
exhaustive bf16 round trips, a library's bf16 rounding, quantisation error
bounds and end points, hand-derived layout words, one-hot and brute-force
products, closed forms of softmax, RMSNorm, RoPE and SiLU."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(h):
    return synth.bf16_to_f32(h).astype(np.float64)


# ------------------------------------------------------------------ bf16 --
def test_bf16_exhaustive_round_trip():
    L = oracle.lib()
    for h in range(1 << 16):
        if (h & 0x7F80) == 0x7F80 and (h & 0x7F):
            continue  # NaN payloads
        f = L.orc_f32_from_bf16(h)
        assert L.orc_bf16_from_f32(f) == h


def test_bf16_rne_matches_torch_and_hand_cases():
    rng = np.random.default_rng(0)
    base = rng.standard_normal(4000).astype(np.float32)
    # exact halfway points between neighbouring bf16 values, both parities
    bits = (base.view(np.uint32) & 0xFFFF0000) | 0x8000
    x = np.concatenate([base, bits.view(np.float32), np.float32([1e-40, -3e38, 0.0, -0.0])])
    ours = oracle.bf16_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa
    assert oracle.bf16_from_f32(np.float32([1 + 2 ** -8]))[0] == 0x3F80
    assert oracle.bf16_from_f32(np.float32([1 + 3 * 2 ** -8]))[0] == 0x3F82
    assert oracle.bf16_from_f32(np.float32([1 + 2 ** -8 + 2 ** -20]))[0] == 0x3F81


# ------------------------------------------------------------- int8 -------
def _w(shape, seed=0, tid=77, sigma=0.02):
    return synth.normal_bf16(seed, tid, shape, sigma)


def test_quant_w8_bound_and_end_points():
    W = _w((96, 4096))
    W[3] = 0                                   # all-zero row
    W[5] = 0
    W[5, 17] = synth.normal_bf16(1, 1, (1,), 1.0)[0]   # single non-zero
    q, s = oracle.quant_w8(W)
    Wd, sd = f32(W), f32(s)
    err = np.abs(Wd - q.astype(np.float64) * sd[:, None])
    assert np.all(err <= sd[:, None] / 2 * (1 + 2e-5))
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    mx = np.abs(Wd).max(axis=1)
    nz = mx > 0
    # bf16 rounding keeps 127*s within 2^-8 of the row maximum
    assert np.all(np.abs(127 * sd[nz] - mx[nz]) <= mx[nz] * 2 ** -8)
    # the largest |w| of each row maps to +-127
    amax = np.abs(Wd).argmax(axis=1)
    assert np.all(np.abs(q[nz, amax[nz]].astype(np.int32)) == 127)
    assert s[3] == 0 and not q[3].any()
    assert q[5, 17] in (127, -127) and np.count_nonzero(q[5]) == 1


def test_quant_w8_codes_are_nearest():
    """Brute force: every code is a nearest integer to w/s (ties either way)."""
    W = _w((8, 512), tid=78)
    q, s = oracle.quant_w8(W)
    Wd, sd = f32(W), f32(s)
    for n in range(8):
        for k in range(0, 512, 7):
            t = Wd[n, k] / sd[n]
            assert abs(q[n, k] - t) <= 0.5 + 1e-5


# ------------------------------------------------------------- int4 -------
def test_quant_w4g_bound_and_end_points():
    W = _w((64, 1024), tid=79)
    W[2, 64:96] = W[2, 70]                       # degenerate group: all equal
    W[4, 0:32] = np.where(np.arange(32) % 2 == 0, W[4, 0], W[4, 1])  # two values
    q, s, z = oracle.quant_w4g(W)
    Wd = f32(W)
    sd = np.repeat(f32(s), 32, axis=1)
    zd = np.repeat(f32(z), 32, axis=1)
    What = q.astype(np.float64) * sd + zd
    assert np.all(np.abs(Wd - What) <= sd / 2 * (1 + 1e-5))
    assert q.max() <= 15
    g = Wd.reshape(64, 32, 32)
    qg = q.reshape(64, 32, 32)
    # z is the group minimum, exactly; the minimum gets code 0, the maximum 15
    assert np.array_equal(f32(z), g.min(axis=2))
    nondeg = g.max(axis=2) > g.min(axis=2)
    amin, amax = g.argmin(axis=2), g.argmax(axis=2)
    ii, jj = np.nonzero(nondeg)
    assert np.all(qg[ii, jj, amin[ii, jj]] == 0)
    assert np.all(qg[ii, jj, amax[ii, jj]] == 15)
    # degenerate group dequantises exactly
    assert s[2, 2] == 0 and np.array_equal(What[2, 64:96], Wd[2, 64:96])
    # a two-valued group uses only the end codes and is exact
    assert set(np.unique(q[4, 0:32])) <= {0, 15}
    assert np.allclose(What[4, 0:32], Wd[4, 0:32], rtol=0, atol=float(sd[4, 0]) * 0.04)


def test_quant_w4g_worked_example():
    """Row k/16 for k = 0..31 (all bf16-exact).  min 0, max 31/16;
    (31/16)/15 = 0.129166..., whose nearest bf16 is 0.12890625 (0x3E04);
    code k = rint(k/16 / 0.12890625) = rint(k * 0.48484848...)."""
    vals = np.arange(32, dtype=np.float32) / 16
    W = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(1, 32)
    q, s, z = oracle.quant_w4g(W)
    assert s[0, 0] == 0x3E04 and z[0, 0] == 0
    expect = [int(round(k * 0.484848484848)) for k in range(32)]
    # k*0.4848 is never within 1e-3 of a .5 boundary here, so Python's round is safe
    assert list(q[0]) == expect


# ------------------------------------------------------------ layout ------
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "layout_chunks.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                parts = line.split()
                words = []
                for p in parts[4:]:
                    if "*" in p:
                        n, v = p.split("*")
                        words += [int(v, 0)] * int(n)
                    else:
                        words.append(int(p, 0))
                rows.append((parts[0], int(parts[1]), int(parts[2]), int(parts[3]), words))
    return rows


def test_layout_hand_words():
    rows = _golden_rows()
    assert [r[0] for r in rows] == ["int4", "int4", "int8"]
    for kind, N, K, G, words in rows:
        if kind == "int4":
            codes = ((np.arange(K)[None, :] + np.arange(N)[:, None]) % 16).astype(np.uint8)
            if G == 32:
                s = np.full((N, K // G), 0x3E04, np.uint16)
                z = np.zeros((N, K // G), np.uint16)
            else:
                s = (0x3C00 + np.arange(N)[:, None] + np.zeros((1, K // G), np.int64)).astype(np.uint16)
                z = (0xBC00 + np.arange(N)[:, None] + np.zeros((1, K // G), np.int64)).astype(np.uint16)
            packed = oracle.pack(oracle.INT4, N, K, codes, s, z, G=G)
        else:
            codes = np.array([-1, 2, -3, 4] * (N * K // 4), np.int8).reshape(N, K)
            packed = oracle.pack(oracle.INT8, N, K, codes)
        assert list(packed.view("<u4")) == words


def _subnormal_decode_int4(word):
    """Decode one packed int4 word the way the GEMV reads it: code i sits in
    bits p..p+3 of the word (i < 6, p = 4i) or of the word shifted right by 8
    bits (i = 6, 7: p = 16, 20); masking those bits and reading the result as
    an IEEE binary32 gives the exact value code * 2^(p - 149) (a subnormal,
    or for bit 23 set the smallest normal binade, which continues it)."""
    out = []
    for i in range(8):
        v, p = (word, 4 * i) if i < 6 else (word >> 8, 4 * i - 8)
        f = np.array([v & (15 << p)], dtype=np.uint32).view(np.float32)[0]
        q = float(f) * 2.0 ** (149 - p)
        assert q == int(q)
        out.append(int(q))
    return out


def _subnormal_decode_int8(word):
    """int8 as the GEMV reads it: byte i is the offset code q + 128, in bits
    p..p+7 of the word (i < 3, p = 8i) or of the word shifted right by 8
    (i = 3, p = 16), read as binary32."""
    out = []
    for i in range(4):
        v, p = (word, 8 * i) if i < 3 else (word >> 8, 16)
        f = np.array([v & (255 << p)], dtype=np.uint32).view(np.float32)[0]
        out.append(int(float(f) * 2.0 ** (149 - p)) - 128)
    return out


def _unswizzle(words, line):
    """The 32 words of slot line `line`, with its 16-byte units put back in
    order (unit u is stored at unit u XOR (line mod 8))."""
    raw = words[line * 32:(line + 1) * 32].reshape(8, 4)
    return np.concatenate([raw[u ^ (line % 8)] for u in range(8)])


def test_layout_views_recover_codes():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    s = rng.integers(0, 1 << 16, size=(3, 2)).astype(np.uint16)
    z = rng.integers(0, 1 << 16, size=(3, 2)).astype(np.uint16)
    packed = oracle.pack(oracle.INT4, 3, 64, codes, s, z)
    words = packed.view("<u4")
    # one slot: row r's 32 code bytes open line r; the scale lines start at
    # line 64, group g's line holding row r's word r
    for r in range(3):
        line = _unswizzle(words, r)
        got = []
        for j in range(8):
            got += _subnormal_decode_int4(int(line[j]))
        assert got == list(codes[r])
    for g in range(2):
        line = _unswizzle(words, 64 + g)
        assert list(line[:3] & 0xFFFF) == list(s[:, g]) and list(line[:3] >> 16) == list(z[:, g])
        assert not line[3:].any()
    codes8 = rng.integers(-127, 128, size=(2, 32)).astype(np.int8)
    words8 = oracle.pack(oracle.INT8, 2, 32, codes8).view("<u4")
    got8 = [c for r in range(2) for w in _unswizzle(words8, r)[:8] for c in _subnormal_decode_int8(int(w))]
    assert got8 == list(codes8.reshape(-1))


@pytest.mark.parametrize("dt,N,K,G", [(0, 45, 8 * 40, 32), (1, 70, 16 * 37, 32), (2, 33, 32 * 45, 32),
                                      (2, 64, 4096, 32), (2, 45, 128 * 3, 128), (2, 7, 64 * 5, 64),
                                      (1, 1, 16, 32), (0, 31, 8, 32)])
def test_layout_bijection(dt, N, K, G):
    rng = np.random.default_rng(dt * 1000 + N)
    if dt == 0:
        src = rng.integers(0, 1 << 16, size=(N, K)).astype(np.uint16)
    elif dt == 1:
        src = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    else:
        src = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    s = z = None
    if dt == 2:
        s = rng.integers(0, 1 << 16, size=(N, K // G)).astype(np.uint16)
        z = rng.integers(0, 1 << 16, size=(N, K // G)).astype(np.uint16)
    packed = oracle.pack(dt, N, K, src, s, z, G=G)
    back, s2, z2 = oracle.unpack(dt, N, K, packed, G=G)
    assert np.array_equal(back, src)
    if dt == 2:
        assert np.array_equal(s2, s) and np.array_equal(z2, z)
    # slots of 32 rows x 256 code bytes (+ 512 / G scale lines of 128 bytes
    # for int4), the ragged tile and K-slot padded
    rowb = K * 2 if dt == 0 else K if dt == 1 else K // 2
    slot = 8192 + ((512 // G) * 128 if dt == 2 else 0)
    assert packed.size == -(-N // 32) * -(-rowb // 256) * slot
    # every code byte of the matrix lands in a distinct byte; the rest is zero
    nz = np.count_nonzero(packed)
    assert nz <= N * rowb + (N * (K // G) * 4 if dt == 2 else 0)


# ------------------------------------------------------------ linear ------
@pytest.mark.parametrize("dt", [0, 1, 2])
def test_linear_one_hot_recovers_columns(dt):
    W = _w((40, 256), tid=90 + dt)
    q, s, z = (W, None, None) if dt == 0 else (oracle.quant_w8(W) + (None,)) if dt == 1 else oracle.quant_w4g(W)
    What = oracle.dequant(dt, q, s, z)
    for j in (0, 31, 32, 200, 255):
        x = np.zeros(256)
        x[j] = 1.0
        y = oracle.linear(dt, q, s, z, x)
        assert np.array_equal(y, What[:, j])


def test_linear_brute_force_tiny():
    from fractions import Fraction
    W = _w((5, 64), tid=95)
    x = synth.bf16_to_f32(synth.normal_bf16(0, 96, (64,))).astype(np.float64)
    q, s, z = oracle.quant_w4g(W)
    y = oracle.linear(2, q, s, z, x)
    for n in range(5):
        exact = Fraction(0)
        for k in range(64):
            g = k // 32
            wk = Fraction(int(q[n, k])) * Fraction(float(f32(s[n, g]))) + Fraction(float(f32(z[n, g])))
            exact += Fraction(float(x[k])) * wk
        assert abs(float(exact) - y[n]) <= 1e-12 * (1 + abs(float(exact)))
    # T rows at once equal T single rows
    X = np.stack([x, -x, 2 * x])
    Y = oracle.linear(2, q, s, z, X)
    assert np.allclose(Y[1], -y, rtol=0, atol=1e-12) and np.allclose(Y[2], 2 * y, rtol=0, atol=1e-12)


# --------------------------------------------------------- attention ------
def test_attention_single_position_returns_v():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((2, 1, 16))
    V = rng.standard_normal((2, 1, 16))
    o = oracle.attention(q, K, V)
    for h in range(4):
        assert np.allclose(o[h], V[h // 2, 0], rtol=0, atol=1e-15)


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 8))
    K = np.repeat(rng.standard_normal((1, 1, 8)), 7, axis=1)
    V = rng.standard_normal((1, 7, 8))
    o = oracle.attention(q, K, V)
    assert np.allclose(o, np.broadcast_to(V[0].mean(axis=0), (2, 8)), atol=1e-14)


def test_attention_brute_force_gqa():
    rng = np.random.default_rng(4)
    Hq, Hkv, hd, T = 6, 2, 8, 5
    q = rng.standard_normal((Hq, hd))
    K = rng.standard_normal((Hkv, T, hd))
    V = rng.standard_normal((Hkv, T, hd))
    o = oracle.attention(q, K, V)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        sc = [sum(q[h, d] * K[g, t, d] for d in range(hd)) / math.sqrt(hd) for t in range(T)]
        e = [math.exp(v) for v in sc]           # no max subtraction: small values
        tot = sum(e)
        for d in range(hd):
            ref = sum(e[t] * V[g, t, d] for t in range(T)) / tot
            assert abs(ref - o[h, d]) < 1e-12


def test_attention_two_keys_closed_form():
    hd = 4
    q = np.array([[1.0, 0, 0, 0]])
    K = np.array([[[2.0, 0, 0, 0], [0.0, 0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0], [0.0, 1, 0, 0]]])
    o = oracle.attention(q, K, V)
    w0 = 1 / (1 + math.exp(-2 / math.sqrt(hd)))   # softmax of (1, 0)
    assert abs(o[0, 0] - w0) < 1e-15 and abs(o[0, 1] - (1 - w0)) < 1e-15


# -------------------------------------------------------- elementwise -----
def test_rmsnorm_constant_input_closed_form():
    g = synth.normal_bf16(0, 97, (64,), 0.02, mu=1.0)
    for c in (0.5, -3.0, 1e-3):
        y = oracle.rmsnorm(np.full(64, c), g, 1e-5)
        ref = f32(g) * c / math.sqrt(c * c + 1e-5)
        assert np.allclose(y, ref, rtol=1e-15, atol=0)


def test_rope_identity_rotation_and_relative_position():
    rng = np.random.default_rng(5)
    hd, H = 16, 3
    v = rng.standard_normal(H * hd)
    assert np.array_equal(oracle.rope(v, H, hd, 0, 1e4), v)
    p = 7
    r = oracle.rope(v, H, hd, p, 1e4)
    # pair 0 turns by exactly p radians (frequency theta^0 = 1)
    x0, x1 = v[0], v[1]
    assert abs(r[0] - (x0 * math.cos(p) - x1 * math.sin(p))) <= 1e-15
    assert abs(r[1] - (x0 * math.sin(p) + x1 * math.cos(p))) <= 1e-15
    # the last pair of a head turns by p * theta^(-2(hd/2-1)/hd)
    f = 1e4 ** (-2.0 * (hd // 2 - 1) / hd)
    y0, y1 = v[hd - 2], v[hd - 1]
    assert abs(r[hd - 2] - (y0 * math.cos(p * f) - y1 * math.sin(p * f))) <= 1e-15
    # each pair keeps its length
    a = v.reshape(-1, 2)
    b = r.reshape(-1, 2)
    assert np.allclose(np.hypot(a[:, 0], a[:, 1]), np.hypot(b[:, 0], b[:, 1]), rtol=1e-14)
    # <R(p)q, R(p')k> depends on p - p' only
    q = rng.standard_normal(hd)
    k = rng.standard_normal(hd)
    d1 = np.dot(oracle.rope(q, 1, hd, 10, 1e4), oracle.rope(k, 1, hd, 4, 1e4))
    d2 = np.dot(oracle.rope(q, 1, hd, 106, 1e4), oracle.rope(k, 1, hd, 100, 1e4))
    assert abs(d1 - d2) < 0.05 * (1 + abs(d1))


def test_swiglu_closed_forms():
    g = np.array([0.0, 1.0, 30.0, -30.0])
    u = np.array([5.0, 2.0, 0.5, 1.0])
    h = oracle.swiglu(g, u)
    assert h[0] == 0.0
    assert abs(h[1] - 2.0 / (1 + math.exp(-1))) < 1e-15
    assert abs(h[2] - 15.0) < 1e-11      # silu(30) = 30 (1 - 9e-14)
    assert abs(h[3]) < 1e-11
