"""Pins of the oracle's exact mode (wide 16-bit weights against int8
per-token activations; BitExact LLM post, "Three execution paths"): the
128-bit requantisation against exact rationals, the wide artifact's relation
to the int8 one, agreement with the float64 restatement of the real-valued
decoder on the wide weights, the fidelity the wide weights add over their
int8 rounding, the prefill / decode invariance at tolerance 0, and a stored
regression fixture written by tests/golden/make_golden.py (oracle only)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import float_model
import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_w16_seed0.json")


@pytest.fixture(scope="module")
def wide_artifact():
    return synth.ensure_artifact("tiny", 0, wide=True)


def _round_half_up(fr: Fraction) -> int:
    # nearest integer, ties toward +infinity
    return (fr + Fraction(1, 2)).__floor__()


def test_requant_wide_is_one_exact_rounding():
    rng = np.random.default_rng(7)
    n = 4000
    acc = rng.integers(-(1 << 35), 1 << 35, n, dtype=np.int64)
    mt = rng.integers(1 << 14, (1 << 15) + 1, n).astype(np.int32)
    mc = rng.integers(1 << 14, 1 << 15, n).astype(np.int32)
    kt = rng.integers(-2, 40, n).astype(np.int32)
    f_out = 16
    # exact ties: acc * mt * mc an odd multiple of 2^(s-1)
    for i in range(200):
        s = int(kt[i]) + 30 - f_out
        mt[i], mc[i] = 1 << 14, 1 << 14
        acc[i] = (2 * i + 1) * (1 << max(0, s - 29)) * (-1 if i % 2 else 1)
    got = oracle.requant_wide(acc, mt, kt, mc, f_out)
    for i in range(n):
        s = int(kt[i]) + 30 - f_out
        want = _round_half_up(Fraction(int(acc[i]) * int(mt[i]) * int(mc[i]), 1 << s))
        assert int(got[i]) == want, (i, int(acc[i]), int(mt[i]), int(mc[i]), s)


def test_requant_wide_beyond_int64_products():
    # acc * m_t * m_c above 2^63: only a 128-bit product gets these right
    acc = np.array([(1 << 35) - 1, -(1 << 35) + 1, (1 << 34) + 12345], np.int64)
    got = oracle.requant_wide(acc, 1 << 15, 30, (1 << 15) - 1, 16)
    for a, g in zip(acc, got):
        want = _round_half_up(Fraction(int(a) * (1 << 15) * ((1 << 15) - 1), 1 << 44))
        assert int(g) == want


def test_wide_artifact_rounds_to_the_int8_artifact(tiny_artifact, wide_artifact):
    a8 = float_model.load(tiny_artifact)
    a16 = float_model.load(wide_artifact)
    assert a16["kc"] == 30 and a8["kc"] == 22

    def check(w16, w8):
        assert w16.dtype == np.int16 and w8.dtype == np.int8
        r = w16.astype(np.int64) - 256 * w8.astype(np.int64)
        assert r.min() >= -127 and r.max() <= 127             # round(w16 / 256) == w8
        assert np.unique(r).size > 200                          # the fine bits are really there

    check(a16["embed"], a8["embed"])
    assert np.array_equal(a16["embed_m"], a8["embed_m"])
    for l16, l8 in zip(a16["layers"], a8["layers"]):
        for k in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
            check(l16[k], l8[k])
        for k in ("m_qkv", "m_o", "m_gate", "m_up", "m_down", "attn_gamma", "ffn_gamma", "q_gamma",
                  "k_gamma", "kvp"):
            assert np.array_equal(l16[k], l8[k]), k


def _rel_errors(path, art, ids):
    lf = float_model.forward(art, ids)
    m = oracle.Model(path)
    s = m.new_seq(64)
    out = []
    for t in range(len(ids)):
        _, lg = s.feed(ids[t:t + 1])
        out.append(np.linalg.norm(lg / 65536.0 - lf[t]) / np.linalg.norm(lf[t]))
    return np.array(out)


@pytest.mark.parametrize("prompt_index", [0, 1, 2])
def test_wide_oracle_tracks_float64_model_closer_than_int8(tiny_artifact, wide_artifact, prompt_index):
    art = float_model.load(wide_artifact)
    ids = synth.prompt_ids(0, prompt_index, 24, art["V"])
    e16 = _rel_errors(wide_artifact, art, ids)
    e8 = _rel_errors(tiny_artifact, art, ids)    # the same real-valued model, weights rounded to int8
    # composition: a transposed operand or a wrong scale shift gives > 25 %
    assert e16.max() < 0.15, e16
    # fidelity: measured ~0.055-0.060 against ~0.081-0.091 for the int8 rounding
    assert e16.mean() < 0.8 * e8.mean(), (e16.mean(), e8.mean())


def test_wide_prefill_equals_token_by_token(wide_artifact):
    m = oracle.Model(wide_artifact)
    assert m.wbits == 16
    ids = synth.prompt_ids(0, 3, 40, m.vocab)
    a = m.new_seq(64)
    am_a, lg_a = a.feed(ids)
    for split in [1, 13, 39]:
        b = m.new_seq(64)
        b.feed(ids[:split])
        for t in range(split, len(ids)):
            am_b, lg_b = b.feed(ids[t:t + 1])
        assert am_a == am_b and np.array_equal(lg_a, lg_b)


def test_wide_golden_regression(wide_artifact):
    with open(GOLDEN) as f:
        g = json.load(f)
    assert open(wide_artifact + ".sha256").read().strip() == g["artifact_sha256"]
    m = oracle.Model(wide_artifact)
    ids = synth.prompt_ids(g["seed"], 0, g["prompt_len"], m.vocab)
    s = m.new_seq(64)
    am, lg = s.feed(ids)
    rows, toks = [lg], [am]
    for _ in range(g["steps"] - 1):
        am, lg = s.feed([toks[-1]])
        rows.append(lg)
        toks.append(am)
    assert toks == g["tokens"]
    assert oracle.chain_hash(rows).hex()[:12] == g["logits_hash12"]


@pytest.mark.slow
def test_wide_no_bound_violation_qwen_shape():
    # every asserted bound of the 16-bit weight path (accumulator < 2^36,
    # shift range, 128-bit product, saturations) on the Qwen3-0.6B shape
    path = synth.ensure_artifact("qwen3-0.6b", 0, wide=True)
    m = oracle.Model(path)
    assert m.wbits == 16
    ids = synth.prompt_ids(0, 0, 6, m.vocab)
    s = m.new_seq(16)
    am, lg, hid = s.feed(ids, want_hidden=True)
    assert np.abs(hid.astype(np.int64)).max() < 2 ** 30
    am2, _ = s.feed([am])
    assert 0 <= am2 < m.vocab
