"""GPU parity of the whole integer forward pass against the CPU oracle at
tolerance 0 (logits of every step, tokens, chain hashes), plus the pages'
invariances on the GPU itself: batch composition, split prefill, graph vs no
graph, repeats (DetLLM README, "Demo"; DetLLM blog footnote on the
zero-tolerance suite)."""
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


def _oracle_run(path, prompt, steps, max_ctx):
    import oracle
    m = oracle.Model(path)
    s = m.new_seq(max_ctx)
    am, lg = s.feed(prompt)
    toks, rows = [am], [lg]
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        toks.append(am)
        rows.append(lg)
    return np.array(toks, np.int32), rows


def _load(path, max_batch, max_ctx):
    import deterministic_integer_only_gb300 as pkg
    return pkg.Model(path, max_batch=max_batch, max_ctx=max_ctx)


@pytest.mark.parametrize("graph,fused", [(True, True), (False, True), (True, False), (False, False)])
def test_tiny_matches_oracle_every_step(torch_cuda, tiny_artifact, graph, fused):
    prompt = synth.prompt_ids(0, 0, 16, 1024)
    ot, orows = _oracle_run(tiny_artifact, prompt, 16, 64)
    if True:
        m = _load(tiny_artifact, 2, 64)
        m.set_graph(graph)
        m.set_fused_decode(fused)
        toks, rows = m.generate([prompt], 16)
        assert np.array_equal(toks[0], ot)
        for s in range(16):
            assert np.array_equal(rows[s][0], orows[s]), f"step {s} graph={graph}"
        assert not m.status().any()
        m.close()


def test_tiny_golden_hash(torch_cuda, tiny_artifact):
    import json
    import os
    import deterministic_integer_only_gb300 as pkg
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_seed0.json")))
    prompt = synth.prompt_ids(g["seed"], 0, g["prompt_len"], 1024)
    m = _load(tiny_artifact, 1, 64)
    toks, rows = m.generate([prompt], g["steps"])
    assert toks[0].tolist() == g["tokens"]
    assert pkg.chain_hash([r[0] for r in rows]).hex()[:12] == g["logits_hash12"]


def test_tiny_batch_composition_and_split_prefill(torch_cuda, tiny_artifact):
    prompt = synth.prompt_ids(0, 0, 16, 1024)
    ot, orows = _oracle_run(tiny_artifact, prompt, 12, 128)
    lens = synth.coprompt_lengths(0, 7, 16, 100)
    cos = [synth.prompt_ids(0, 100 + i, int(n), 1024) for i, n in enumerate(lens)]
    m = _load(tiny_artifact, 8, 128)
    toks, rows = m.generate([prompt] + cos, 12)
    assert np.array_equal(toks[0], ot)
    for s in range(12):
        assert np.array_equal(rows[s][0], orows[s])
    # a co-prompt row matches the oracle too
    ot3, orows3 = _oracle_run(tiny_artifact, cos[3], 12, 128)
    assert np.array_equal(toks[4], ot3)
    assert all(np.array_equal(rows[s][4], orows3[s]) for s in range(12))
    m.close()
    # split prefill: 7 tokens at once, the rest one by one, then decode
    torch = torch_cuda
    m = _load(tiny_artifact, 1, 128)
    dev = torch.device("cuda")
    lg = torch.empty((1, 1024), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        m.prefill([0], torch.tensor(prompt[:7], device=dev), [0, 7], lg, tok)
        for t in prompt[7:]:
            m.decode_step([0], torch.tensor([t], dtype=torch.int32, device=dev), lg, tok)
        out = [int(tok.item())]
        rows2 = [lg.cpu().numpy()[0]]
        for _ in range(11):
            m.decode_step([0], tok, lg, tok)
            out.append(int(tok.item()))
            rows2.append(lg.cpu().numpy()[0])
    assert out == ot.tolist()
    assert all(np.array_equal(a, b) for a, b in zip(rows2, orows))
    m.close()


def test_tiny_repeats_and_reset(torch_cuda, tiny_artifact):
    prompt = synth.prompt_ids(0, 5, 20, 1024)
    m = _load(tiny_artifact, 1, 64)
    ref = None
    for _ in range(3):
        toks, rows = m.generate([prompt], 8, keep_logits="hash")
        if ref is None:
            ref = (toks, rows)
        assert np.array_equal(toks, ref[0]) and rows == ref[1]
        m.reset_seq(0)
    m.close()


def test_bad_inputs_are_reported(torch_cuda, tiny_artifact):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    m = _load(tiny_artifact, 2, 32)
    dev = torch.device("cuda")
    with pytest.raises(pkg.DetintError) as e:
        m.prefill([5], torch.zeros(4, dtype=torch.int32, device=dev), [0, 4])
    assert e.value.code == 9
    with pytest.raises(pkg.DetintError) as e:
        m.prefill([0], torch.zeros(40, dtype=torch.int32, device=dev), [0, 40])
    assert e.value.code == 4
    with torch.cuda.stream(m.stream):
        m.prefill([1], torch.tensor([3, 2000, 7], dtype=torch.int32, device=dev), [0, 3])
    flags = m.status()
    assert flags[0] == 1
    m.close()


@pytest.mark.parametrize("fused", [True, False])
def test_qwen_shape_matches_oracle(torch_cuda, qwen_artifact, fused):
    prompt = synth.prompt_ids(0, 0, 64, 151936)
    ot, orows = _oracle_run(qwen_artifact, prompt, 6, 128)
    m = _load(qwen_artifact, 8, 1024)
    m.set_fused_decode(fused)
    toks, rows = m.generate([prompt], 6)
    assert np.array_equal(toks[0], ot)
    for s in range(6):
        assert np.array_equal(rows[s][0], orows[s]), f"step {s}"
    assert not m.status().any()
    m.close()


def test_qwen_batch8_row0_equals_batch1(torch_cuda, qwen_artifact):
    prompt = synth.prompt_ids(0, 0, 64, 151936)
    lens = synth.coprompt_lengths(0, 7)
    cos = [synth.prompt_ids(0, 100 + i, int(n), 151936) for i, n in enumerate(lens)]
    m = _load(qwen_artifact, 8, 1024)
    t1, h1 = m.generate([prompt], 24, keep_logits="hash")
    m.reset_seq(0)
    t8, h8 = m.generate([prompt] + cos, 24, keep_logits="hash")
    assert np.array_equal(t8[0], t1[0]) and h8[0] == h1[0]
    m.close()


@pytest.mark.parametrize("B", [2, 3, 4, 5, 8])
def test_tiny_batch_sizes_match_oracle(torch_cuda, tiny_artifact, B):
    """Decode batches of 2 (quantisation fused into the GEMV prologue) and
    of 3 to 8 (rows quantised by the row kernels) agree with the oracle."""
    prompts = [synth.prompt_ids(7, i, 10 + 4 * i, 1024) for i in range(B)]
    m = _load(tiny_artifact, B, 64)
    toks, rows = m.generate(prompts, 6)
    for b in (0, B - 1):
        ot, orows = _oracle_run(tiny_artifact, prompts[b], 6, 64)
        assert np.array_equal(toks[b], ot)
        assert all(np.array_equal(rows[s][b], orows[s]) for s in range(6))
    m.close()


@pytest.mark.parametrize("name", ["qwen", "llama"])
def test_staged_decode_attention_equals_per_token(torch_cuda, request, name):
    """The decode attention that stages the cached K/V in shared memory gives
    the per-token kernel's logits: a batch of 3 ragged prompts, 24 steps."""
    path = request.getfixturevalue({"qwen": "qwen_artifact", "llama": "llama_artifact"}[name])
    V = {"qwen": 151936, "llama": 128256}[name]
    prompts = [synth.prompt_ids(8, i, n, V) for i, n in enumerate((5, 64, 190))]
    out = {}
    for staged in (True, False):
        m = _load(path, 4, 512)
        m.set_staged_decode(staged)
        out[staged] = m.generate(prompts, 24, keep_logits="hash")
        m.close()
    assert np.array_equal(out[True][0], out[False][0])
    assert out[True][1] == out[False][1]


def test_staged_decode_capacity_crossing(torch_cuda, qwen_artifact):
    """A context that grows past the staged capacity (768 keys at this shape)
    mid-generation switches kernels without changing a logit."""
    prompt = synth.prompt_ids(8, 9, 760, 151936)
    out = {}
    for staged in (True, False):
        m = _load(qwen_artifact, 1, 1024)
        m.set_staged_decode(staged)
        out[staged] = m.generate([prompt], 16, keep_logits="hash")
        m.close()
    assert np.array_equal(out[True][0], out[False][0])
    assert out[True][1] == out[False][1]


@pytest.mark.parametrize("name", ["tiny", "qwen", "llama"])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_persistent_decode_equals_kernel_chain(torch_cuda, request, name, B):
    """The one-launch decode step (cooperative grid, phases handed over
    through tagged activation words) gives the kernel chain's logits and
    tokens, batch of B."""
    path = request.getfixturevalue({"tiny": "tiny_artifact", "qwen": "qwen_artifact",
                                    "llama": "llama_artifact"}[name])
    V = {"tiny": 1024, "qwen": 151936, "llama": 128256}[name]
    prompts = [synth.prompt_ids(12, i, n, V) for i, n in enumerate((9, 70, 33, 5, 128, 17, 64, 40)[:B])]
    out = {}
    for pers in (True, False):
        m = _load(path, 8, 256)
        m.set_persistent(pers)
        out[pers] = m.generate(prompts, 12, keep_logits="hash")
        assert not m.status().any()
        m.close()
    assert np.array_equal(out[True][0], out[False][0])
    assert out[True][1] == out[False][1]


@pytest.mark.parametrize("graph", [True, False])
def test_decode_step_wait_timeout_is_reported_and_recovers(torch_cuda, tiny_artifact, graph):
    """Failure path of the bounded waits: with the wait test on, the one-launch
    step's final wait expects a tag that no CTA writes, gives up after a few
    thousand polls and records status slot 6 instead of hanging. The step's
    logits (written before that wait) still equal the oracle's, and once the
    test is off the sequence continues exactly as the oracle does."""
    torch = torch_cuda
    dev = torch.device("cuda")
    prompt = synth.prompt_ids(4, 0, 16, 1024)
    ot, orows = _oracle_run(tiny_artifact, prompt, 8, 64)
    m = _load(tiny_artifact, 2, 64)
    m.set_graph(graph)
    m.set_persistent(True)
    lg = torch.empty((1, 1024), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        m.prefill([0], torch.tensor(prompt, dtype=torch.int32, device=dev), [0, len(prompt)], lg, tok)
    assert not m.status().any()
    for step in range(1, 8):
        stall = step == 3
        m.set_wait_test(2000 if stall else 0)
        fed = torch.tensor([int(ot[step - 1])], dtype=torch.int32, device=dev)
        with torch.cuda.stream(m.stream):
            m.decode_step([0], fed, lg, tok)
        st = m.status()
        assert np.array_equal(lg.cpu().numpy()[0], orows[step]), step
        if stall:
            assert st[6] == 1 and st[:6].sum() == 0
        else:
            assert not st.any(), step
            assert int(tok.item()) == int(ot[step]), step
    m.close()
