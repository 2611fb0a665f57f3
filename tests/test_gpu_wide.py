"""Exact mode (16-bit weights) on the GPU: the BitExact LLM post's exact mode
keeps the linear layers' wide weights against fixed-point activations
("Three execution paths"), multiplying them as integer limbs combined in
wider accumulators ("Fix the arithmetic, not just the random seed"). The
library loads a version-2 artifact as two int8 limbs per weight, runs every
GEMM on the exact limb GEMM (int64 accumulators) and requantises through
the 128-bit product; its logits and tokens must equal the CPU oracle's."""
import json
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deterministic_integer_only_gb300 as pkg
    pkg.lib()
    return torch


def _oracle(path, prompt, steps, max_ctx):
    import oracle
    oracle.set_threads(oracle.max_threads())
    s = oracle.Model(path).new_seq(max_ctx)
    am, lg = s.feed(prompt)
    toks, rows = [am], [lg]
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        toks.append(am)
        rows.append(lg)
    return np.array(toks, np.int32), rows


def test_tiny_wide_matches_oracle_golden(torch_cuda):
    """The tiny model's wide artifact: tokens and logits chain hash of the
    oracle's fixture (16-token seeded prompt, 16 greedy steps)."""
    import deterministic_integer_only_gb300 as pkg
    here = os.path.dirname(os.path.abspath(__file__))
    g = json.load(open(os.path.join(here, "golden", "oracle_tiny_w16_seed0.json")))
    path = synth.ensure_artifact("tiny", g["seed"], wide=True)
    assert open(path + ".sha256").read().strip() == g["artifact_sha256"]
    prompt = synth.prompt_ids(g["seed"], 0, g["prompt_len"], 1024)
    for graph in (True, False):
        m = pkg.Model(path, max_batch=2, max_ctx=64)
        m.set_graph(graph)
        toks, rows = m.generate([prompt], g["steps"])
        assert toks[0].tolist() == g["tokens"], graph
        assert pkg.chain_hash([r[0] for r in rows]).hex()[:12] == g["logits_hash12"], graph
        assert not m.status().any()
        m.close()


def test_tiny_wide_batch_and_split_prefill_invariance(torch_cuda):
    """Three sequences decoded together, and a prompt prefilled in two
    pieces, give the oracle's logits row by row (exact mode)."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    dev = torch.device("cuda")
    path = synth.ensure_artifact("tiny", 0, wide=True)
    prompts = [synth.prompt_ids(31, i, n, 1024) for i, n in enumerate((11, 40, 23))]
    m = pkg.Model(path, max_batch=3, max_ctx=96)
    toks, rows = m.generate(prompts, 8)
    for b in range(3):
        ot, orows = _oracle(path, prompts[b], 8, 96)
        assert np.array_equal(toks[b], ot), b
        for st in range(8):
            assert np.array_equal(rows[st][b], orows[st]), (b, st)
    m.reset_seq(0)
    lg = torch.empty((1, 1024), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    p = prompts[1]
    with torch.cuda.stream(m.stream):
        m.prefill([0], torch.tensor(p[:17], dtype=torch.int32, device=dev), [0, 17], lg, tok)
        m.prefill([0], torch.tensor(p[17:], dtype=torch.int32, device=dev), [0, len(p) - 17], lg, tok)
    m.stream.synchronize()
    _, orows = _oracle(path, p, 1, 96)
    assert np.array_equal(lg.cpu().numpy()[0], orows[0])
    m.close()


def test_qwen_shape_wide_matches_oracle(torch_cuda):
    """The Qwen3-0.6B-shaped wide artifact (16-bit weights from the int8
    artifact of the same seed): every logits row of a 16-token prompt and 6
    greedy steps equals the oracle's."""
    import deterministic_integer_only_gb300 as pkg
    path = synth.ensure_artifact("qwen3-0.6b", 0, wide=True)
    prompt = synth.prompt_ids(0, 0, 16, 151936)
    ot, orows = _oracle(path, prompt, 6, 64)
    m = pkg.Model(path, max_batch=1, max_ctx=64)
    toks, rows = m.generate([prompt], 6)
    assert np.array_equal(toks[0], ot)
    for st in range(6):
        assert np.array_equal(rows[st][0], orows[st]), st
    assert not m.status().any()
    m.close()
