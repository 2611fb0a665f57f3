"""Pins of the oracle's integer operators against float64 restatements of the
real-valued operation they approximate, closed forms and special cases
(DetLLM blog, section "DetLLM" and its QK^T footnote; DetLLM README
"Layout": DI-Softmax, DI-RMSNorm, DI-SwiGLU, int RoPE)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from synth.artifact import rope_tables


def _rows(rng, rows, n, bits):
    x = rng.normal(0, 1, size=(rows, n)) * (2.0 ** bits) / 4
    return np.clip(np.rint(x), -(2 ** 31 - 1), 2 ** 31 - 1).astype(np.int32)


@pytest.mark.parametrize("bits", [3, 12, 20, 28, 30])
def test_actquant_rounds_127x_over_max(bits):
    rng = np.random.default_rng(bits)
    x = _rows(rng, 20, 1000, bits)
    q, mt, kt = oracle.actquant(x, 12)
    for r in range(x.shape[0]):
        a = np.abs(x[r].astype(np.int64)).max()
        if a == 0:
            continue
        ideal = 127.0 * x[r].astype(np.float64) / a
        assert np.max(np.abs(q[r] - ideal)) <= 0.5 + 1e-5
        assert np.abs(q[r].astype(np.int64)).max() == 127
        # the dyadic token scale is a/127 on the x grid, to 15 bits
        scale = mt[r] / 2.0 ** kt[r]
        assert abs(scale - a / 127.0 / 2 ** 12) <= 2.0 ** -14 * scale
        assert 2 ** 14 <= mt[r] <= 2 ** 15


def test_actquant_special_rows():
    z = np.zeros((1, 64), np.int32)
    q, mt, kt = oracle.actquant(z, 12)
    assert not q.any() and mt[0] == 0
    one = np.zeros((1, 64), np.int32)
    one[0, 5] = -7
    q, mt, kt = oracle.actquant(one, 12)
    assert q[0, 5] == -127 and np.count_nonzero(q) == 1
    big = np.full((1, 8), 2 ** 31 - 1, np.int32)
    big[0, 1] = -(2 ** 31 - 1)
    q, _, _ = oracle.actquant(big, 16)
    assert q[0, 0] == 127 and q[0, 1] == -127


def _float_rmsnorm(x, gamma, eps):
    xf = x.astype(np.float64) / 2 ** 16
    return xf / np.sqrt(np.mean(xf * xf) + eps) * gamma.astype(np.float64) / 4096


@pytest.mark.parametrize("bits,n", [(10, 256), (20, 1024), (26, 1024), (30, 2048), (16, 64)])
def test_normquant_against_float64_rmsnorm(bits, n):
    rng = np.random.default_rng(bits + n)
    x = _rows(rng, 10, n, bits)
    gamma = rng.integers(2 ** 11, 2 ** 13, size=n).astype(np.int16)
    eps = 1e-6
    q, mt, kt = oracle.normquant(x, gamma, round(eps * 2 ** 32))
    for r in range(x.shape[0]):
        ref = _float_rmsnorm(x[r], gamma, eps)
        deq = q[r].astype(np.float64) * mt[r] / 2.0 ** kt[r]
        # spec bound for the normalisation: 2^-7 of the row maximum
        assert np.max(np.abs(deq - ref)) <= 2.0 ** -7 * np.abs(ref).max()
        assert np.abs(q[r].astype(np.int64)).max() == 127


def test_normquant_zero_and_tiny_rows():
    n = 256
    gamma = np.full(n, 4096, np.int16)
    q, mt, _ = oracle.normquant(np.zeros((1, n), np.int32), gamma, 4295)
    assert not q.any() and mt[0] == 0
    x = np.zeros((1, n), np.int32)
    x[0, :4] = [1, -1, 1, 1]
    q, mt, kt = oracle.normquant(x, gamma, 4295)
    # a row far below eps: the norm output is x/sqrt(eps)-ish, tiny
    ref = _float_rmsnorm(x[0], gamma, 1e-6)
    deq = q[0] * mt[0] / 2.0 ** kt[0]
    assert np.max(np.abs(deq - ref)) <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("bits", [8, 15, 22])
def test_qknorm_against_float64(bits):
    rng = np.random.default_rng(bits)
    d = 128
    x = _rows(rng, 16, d, bits)
    gamma = rng.integers(2 ** 11, 2 ** 13, size=d).astype(np.int16)
    eps = 1e-6
    y = oracle.qknorm(x, gamma, round(eps * 2 ** 24))
    for r in range(x.shape[0]):
        xf = x[r].astype(np.float64) / 2 ** 12
        ref = xf / np.sqrt(np.mean(xf * xf) + eps) * gamma / 4096.0
        got = y[r] / 2.0 ** 14
        assert np.max(np.abs(got - ref)) <= 2.0 ** -12 * np.abs(ref).max() + 2.0 ** -13


def test_rope_tables_match_float64_and_rotation():
    shape = synth.MODEL_SHAPES["tiny"]
    c, s = rope_tables(shape)
    half = shape.head_dim // 2
    for p in [0, 1, 7, 100, shape.max_pos - 1]:
        for i in range(half):
            ang = p * shape.rope_theta ** (-2.0 * i / shape.head_dim)
            assert abs(int(c[p, i]) - 16384 * math.cos(ang)) <= 0.5 + 1e-9
            assert abs(int(s[p, i]) - 16384 * math.sin(ang)) <= 0.5 + 1e-9
    assert c[0].tolist() == [16384] * half and s[0].tolist() == [0] * half
    rng = np.random.default_rng(9)
    y = rng.integers(-(2 ** 18), 2 ** 18, size=shape.head_dim).astype(np.int32)
    for p in [0, 3, 500]:
        out = oracle.rope(y, c[p], s[p])
        a, b = y[:half].astype(np.float64), y[half:].astype(np.float64)
        cf, sf = c[p] / 16384.0, s[p] / 16384.0
        ref = np.concatenate([a * cf - b * sf, b * cf + a * sf])
        assert np.max(np.abs(out - ref)) <= 0.5 + 1e-9
    # position 0 is the identity
    assert np.array_equal(oracle.rope(y, c[0], s[0]), y)


def test_swiglu_against_float64():
    rng = np.random.default_rng(5)
    g = np.clip(rng.normal(0, 6, 20000) * 4096, -(2 ** 24), 2 ** 24).astype(np.int32)
    u = np.clip(rng.normal(0, 6, 20000) * 4096, -(2 ** 24), 2 ** 24).astype(np.int32)
    g[:6] = [0, 1, -1, 2 ** 24, -(2 ** 24), 4096 * 40]
    s = oracle.swiglu(g, u).astype(np.float64) / 2 ** 10
    gf, uf = g / 4096.0, u / 4096.0
    with np.errstate(over="ignore"):
        ref = gf / (1.0 + np.exp(-gf)) * uf
    tol = 2.0 ** -8 * np.abs(gf * uf) + 2.0 ** -9
    assert np.all(np.abs(s - ref) <= tol)


def test_gemm_matches_numpy_brute_force():
    rng = np.random.default_rng(6)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (17, 33, 64), (64, 16, 300)]:
        A = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        B = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
        ref = A.astype(np.int64) @ B.astype(np.int64).T
        assert np.array_equal(oracle.gemm_i8(A, B), ref)
    A = np.full((2, 8192), 127, np.int8)
    B = np.full((3, 8192), -127, np.int8)
    assert oracle.gemm_i8(A, B).min() == -127 * 127 * 8192


def _kvp(d, e=None, cstm=20000, cstk=22, mv=20000, kv=18):
    half = d // 2
    kvp = np.zeros(8 + half, np.int32)
    kvp[4], kvp[5], kvp[6], kvp[7] = mv, kv, cstm, cstk
    if e is not None:
        kvp[8:] = e
    return kvp


def test_attention_probabilities_against_float64_softmax():
    rng = np.random.default_rng(7)
    d = 128
    for ctx in [1, 2, 17, 300, 2048]:
        q8 = rng.integers(-127, 128, d).astype(np.int8)
        K8 = rng.integers(-127, 128, (ctx, d)).astype(np.int8)
        V8 = rng.integers(-127, 128, (ctx, d)).astype(np.int8)
        mq, kq = 20000, 30
        kvp = _kvp(d)
        o, P, sig = oracle.attention_row(q8, mq, kq, K8, V8, kvp)
        S = K8.astype(np.int64) @ q8.astype(np.int64)
        # the logit in base-2 units that the integer path rounds to Q10
        u = S * mq * kvp[6] / 2.0 ** (kq + kvp[7])
        p = np.exp2(u - u.max())
        p /= p.sum()
        assert np.max(np.abs(P / 2.0 ** 15 - p)) <= 2.0 ** -9
        # output: the softmax average of the values, in Q12 of dequantised v
        ref = (p @ V8.astype(np.float64)) * kvp[4] / 2.0 ** kvp[5]
        assert np.max(np.abs(o / 4096.0 - ref)) <= 2.0 ** -8 * 127 * kvp[4] / 2.0 ** kvp[5]


def test_attention_single_key_returns_dequantised_value():
    rng = np.random.default_rng(8)
    d = 64
    v = rng.integers(-127, 128, (1, d)).astype(np.int8)
    k = rng.integers(-127, 128, (1, d)).astype(np.int8)
    q = rng.integers(-127, 128, d).astype(np.int8)
    kvp = _kvp(d, mv=23456, kv=19)
    o, P, sig = oracle.attention_row(q, 17000, 28, k, v, kvp)
    assert sig == 2 ** 15 - 1 and P[0] == 2 ** 15
    for c in range(d):
        exact = Fraction(int(v[0, c]) * 23456 * 4096, 2 ** 19)
        assert abs(exact - int(o[c])) <= Fraction(1, 2)


def test_attention_equal_scores_average_values():
    rng = np.random.default_rng(10)
    d, ctx = 64, 37
    k = np.tile(rng.integers(-127, 128, (1, d)).astype(np.int8), (ctx, 1))
    v = rng.integers(-127, 128, (ctx, d)).astype(np.int8)
    q = rng.integers(-127, 128, d).astype(np.int8)
    kvp = _kvp(d, mv=2 ** 14, kv=14)   # s_v = 1
    o, P, sig = oracle.attention_row(q, 17000, 28, k, v, kvp)
    assert sig == ctx * (2 ** 15 - 1)
    mean = v.astype(np.float64).mean(0)
    assert np.max(np.abs(o / 4096.0 - mean)) <= 1.0 / 4096 + 1e-9


def test_argmax_lowest_index_on_ties():
    rng = np.random.default_rng(11)
    for _ in range(50):
        x = rng.integers(-50, 50, size=1000).astype(np.int32)
        assert oracle.argmax(x) == int(np.argmax(x))   # numpy returns the first maximum
    x = np.zeros(151936, np.int32)
    assert oracle.argmax(x) == 0
    x[[7, 3, 99]] = 5
    assert oracle.argmax(x) == 3
    x[151935] = 6
    assert oracle.argmax(x) == 151935
