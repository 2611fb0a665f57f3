"""GPU parity at the configured workload sizes (the pages' demo: 64-token
prompt, 512 greedy steps, per-step logits chain hash; DetLLM README "Demo"):
the CUDA path against the CPU oracle, run live where it finishes in seconds
and through fixtures the oracle wrote (tests/golden/make_golden.py --full)
where it needs minutes, plus the invariances that hold at any size (batch
composition, split prefill)."""
import json
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sha(path):
    with open(path + ".sha256") as f:
        return f.read().strip()

pytestmark = pytest.mark.gpu

QWEN_V = 151936
LLAMA_V = 128256


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deterministic_integer_only_gb300 as pkg
    pkg.lib()
    return torch


def _oracle_hashes(path, prompt, steps, max_ctx):
    import oracle
    oracle.set_threads(oracle.max_threads())
    m = oracle.Model(path)
    s = m.new_seq(max_ctx)
    am, lg = s.feed(prompt)
    toks, h = [am], oracle.chain_hash([lg])
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        toks.append(am)
        h = oracle.chain_hash([lg], h)
    return np.array(toks, np.int32), h


def test_config2_512_steps_match_oracle(torch_cuda, qwen_artifact):
    """Qwen3-0.6B shape, B=1, 64-token prompt, 512 greedy steps: tokens and
    the 512-row logits chain hash equal the oracle's."""
    import deterministic_integer_only_gb300 as pkg
    prompt = synth.prompt_ids(0, 0, 64, QWEN_V)
    ot, oh = _oracle_hashes(qwen_artifact, prompt, 512, 640)
    m = pkg.Model(qwen_artifact, max_batch=8, max_ctx=640)
    toks, hashes = m.generate([prompt], 512, keep_logits="hash")
    assert np.array_equal(toks[0], ot)
    assert hashes[0] == oh
    assert not m.status().any()
    m.close()


def test_config3_batch8_row0_equals_batch1_512_steps(torch_cuda, qwen_artifact):
    """Batch 8 with seven co-prompts of lengths U[16, 256]: row 0's 512 tokens
    and logits hash equal the batch-1 run (the row-0 reading of config 3)."""
    import deterministic_integer_only_gb300 as pkg
    prompt = synth.prompt_ids(0, 0, 64, QWEN_V)
    lens = synth.coprompt_lengths(0, 7)
    cos = [synth.prompt_ids(0, 100 + i, int(n), QWEN_V) for i, n in enumerate(lens)]
    m = pkg.Model(qwen_artifact, max_batch=8, max_ctx=800)
    t1, h1 = m.generate([prompt], 512, keep_logits="hash")
    m.reset_seq(0)
    t8, h8 = m.generate([prompt] + cos, 512, keep_logits="hash")
    assert np.array_equal(t8[0], t1[0]) and h8[0] == h1[0]
    m.close()


def test_config4_split_prefill_equals_single_pass(torch_cuda, qwen_artifact):
    """2048-token prompt: 1024 prefilled at once and the rest fed one token at
    a time, then 512 decode steps, equals the single 2048-token prefill, and
    both equal the oracle's tokens and logits chain hash (fixture)."""
    import hashlib
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    dev = torch.device("cuda")
    g = _golden("oracle_qwen06b_split2048.json")
    assert g["artifact_sha256"] == _sha(qwen_artifact)
    prompt = synth.prompt_ids(g["prompt_seed"], g["index"], g["prompt_len"], QWEN_V)
    steps = g["steps"]
    m = pkg.Model(qwen_artifact, max_batch=2, max_ctx=2048 + steps)
    lg = torch.empty((1, QWEN_V), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)

    def run(split):
        h = b"\0" * 32
        out = []
        first = None
        with torch.cuda.stream(m.stream):
            if split:
                m.prefill([0], torch.tensor(prompt[:1024], device=dev), [0, 1024], lg, tok)
                for t in prompt[1024:]:
                    m.decode_step([0], torch.tensor([t], dtype=torch.int32, device=dev), lg, tok)
            else:
                m.prefill([0], torch.tensor(prompt, device=dev), [0, 2048], lg, tok)
            for step in range(steps):
                if step:
                    m.decode_step([0], tok, lg, tok)
                out.append(int(tok.item()))
                row = lg.cpu().numpy().astype("<i4").tobytes()
                if first is None:
                    first = hashlib.sha256(b"\0" * 32 + row).hexdigest()[:12]
                h = hashlib.sha256(h + row).digest()
        return out, h.hex()[:12], first

    a = run(False)
    m.reset_seq(0)
    b = run(True)
    assert a == b
    assert a[0] == g["tokens"]
    assert a[1] == g["logits_hash12"]
    assert a[2] == g["prefill_logits_hash12"]
    assert not m.status().any()
    m.close()


def test_prefill_4096_matches_oracle(torch_cuda, qwen_artifact):
    """One 4096-token prefill (the zero-tolerance suite's 4k context: DetLLM
    blog footnote): the last position's logits hash and token equal the
    oracle's token-by-token run (fixture)."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    dev = torch.device("cuda")
    g = _golden("oracle_qwen06b_prefill4096.json")
    assert g["artifact_sha256"] == _sha(qwen_artifact)
    prompt = synth.prompt_ids(g["prompt_seed"], g["index"], g["prompt_len"], QWEN_V)
    m = pkg.Model(qwen_artifact, max_batch=1, max_ctx=4096)
    lg = torch.empty((1, QWEN_V), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        m.prefill([0], torch.tensor(prompt, device=dev), [0, 4096], lg, tok)
    m.stream.synchronize()
    assert int(tok.item()) == g["tokens"][0]
    assert pkg.chain_hash([lg.cpu().numpy()[0]]).hex()[:12] == g["prefill_logits_hash12"]
    assert not m.status().any()
    m.close()


def test_llama_shape_matches_oracle(torch_cuda, llama_artifact):
    """Llama-3.2-1B shape (no QK-norm, head_dim 64, 4 q heads per kv head):
    two sequences, short prompts, 6 greedy steps, every logits row equal to
    the oracle's."""
    import deterministic_integer_only_gb300 as pkg
    import oracle
    prompts = [synth.prompt_ids(5, i, 24 + 9 * i, LLAMA_V) for i in range(2)]
    m = pkg.Model(llama_artifact, max_batch=2, max_ctx=128)
    toks, rows = m.generate(prompts, 6)
    om = oracle.Model(llama_artifact)
    for b in range(2):
        s = om.new_seq(128)
        am, lg = s.feed(prompts[b])
        for step in range(6):
            if step:
                am, lg = s.feed([int(toks[b, step - 1])])
            assert int(toks[b, step]) == am
            assert np.array_equal(rows[step][b], lg), (b, step)
    m.close()


def test_config5_llama_batch32_rows_equal_batch1(torch_cuda, llama_artifact):
    """Llama-3.2-1B shape, batch 32 of 1024-token contexts: sampled rows of
    the batch-32 decode equal batch-1 runs of the same prompts and the
    oracle's tokens and logits chain hash over 16 steps (fixture)."""
    import deterministic_integer_only_gb300 as pkg
    g = _golden("oracle_llama1b_ctx1024.json")
    prompts = [synth.prompt_ids(9, i, 1024, LLAMA_V) for i in range(32)]
    m = pkg.Model(llama_artifact, max_batch=32, max_ctx=1024 + 32)
    t32, h32 = m.generate(prompts, 16, keep_logits="hash")
    for b in (0, 17):
        ref = g["rows"][str(b)]
        assert ref["artifact_sha256"] == _sha(llama_artifact)
        assert t32[b].tolist() == ref["tokens"], b
        assert h32[b].hex()[:12] == ref["logits_hash12"], b
        for sid in range(32):
            m.reset_seq(sid)
        t1, h1 = m.generate([prompts[b]], 16, keep_logits="hash")
        assert np.array_equal(t1[0], t32[b]) and h1[0] == h32[b], b
    m.close()
