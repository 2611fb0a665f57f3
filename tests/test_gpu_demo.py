"""The pages' demo on this library (DetLLM README, "Demo"; DetLLM blog, the
"one prompt, nine configurations, one hash" table): the Qwen3-0.6B-shaped
model, a 64-token seeded prompt, 512 greedy steps, the per-step logits chain
hash — computed under nine execution configurations, each aimed at a
different source of nondeterminism, and compared with the CPU oracle's hash
stored in tests/golden/oracle_qwen06b_demo.json. One hash for all."""
import hashlib
import json
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_qwen06b_demo.json")
V, STEPS = 151936, 512


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deterministic_integer_only_gb300 as pkg
    pkg.lib()
    return torch


def _hash_row0(torch, m, sids, prompts, split=None):
    """Greedy STEPS of row 0 (prefilled whole, or split: first part at once,
    the rest token by token); returns (logits hash12, tokens hash12)."""
    dev = torch.device("cuda")
    B = len(sids)
    lg = torch.empty((B, V), dtype=torch.int32, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    h, ht = b"\0" * 32, b"\0" * 32
    with torch.cuda.stream(m.stream):
        if split is None:
            cu = np.zeros(B + 1, np.int64)
            cu[1:] = np.cumsum([len(p) for p in prompts])
            flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
            m.prefill(sids, flat, cu, lg, tok)
        else:
            p = prompts[0]
            m.prefill(sids, torch.tensor(p[:split], dtype=torch.int32, device=dev), [0, split], lg, tok)
            for t in p[split:]:
                m.decode_step(sids, torch.tensor([t], dtype=torch.int32, device=dev), lg, tok)
        for step in range(STEPS):
            if step:
                m.decode_step(sids, tok, lg, tok)
            h = hashlib.sha256(h + lg[0].cpu().numpy().astype("<i4").tobytes()).digest()
            ht = hashlib.sha256(ht + np.array([int(tok[0].item())], "<i4").tobytes()).digest()
    return h.hex()[:12], ht.hex()[:12]


def test_demo_nine_configurations_one_hash(torch_cuda, qwen_artifact):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    golden = json.load(open(GOLDEN))
    if open(qwen_artifact + ".sha256").read().strip() != golden["artifact_sha256"]:
        pytest.fail("the synthetic artifact differs from the one the golden hash was computed on")
    prompt = synth.prompt_ids(0, 0, 64, V)
    co7 = [synth.prompt_ids(0, 100 + i, int(n), V) for i, n in enumerate(synth.coprompt_lengths(0, 7))]
    co31 = [synth.prompt_ids(0, 200 + i, int(n), V) for i, n in enumerate(synth.coprompt_lengths(1, 31))]
    configs = [
        ("batch 1 (CUDA graph, fused step)", 1, [prompt], None, {}),
        ("batch 1, no CUDA graph", 1, [prompt], None, {"graph": False}),
        ("batch 8, 7 seeded co-prompts", 8, [prompt] + co7, None, {}),
        ("split prefill (32 + 32 token by token)", 1, [prompt], 32, {}),
        ("batch 32, 31 co-prompts (unfused path, tiled GEMMs)", 32, [prompt] + co31, None, {}),
        ("batch 1, row kernels instead of the fused step", 1, [prompt], None, {"fused": False}),
        ("batch 1, one persistent launch per step", 1, [prompt], None, {"persistent": True}),
        ("batch 8, per-token decode attention", 8, [prompt] + co7, None, {"staged": False}),
        ("split prefill, per-token prefill attention", 1, [prompt], 40, {"tc": False}),
    ]
    table = []
    for name, B, prompts, split, opts in configs:
        m = pkg.Model(qwen_artifact, max_batch=B, max_ctx=64 + STEPS + 256 + 64)
        if "graph" in opts:
            m.set_graph(opts["graph"])
        if "fused" in opts:
            m.set_fused_decode(opts["fused"])
        if "persistent" in opts:
            m.set_persistent(opts["persistent"])
        if "staged" in opts:
            m.set_staged_decode(opts["staged"])
        if "tc" in opts:
            m.set_tc_prefill(opts["tc"])
        hl, ht = _hash_row0(torch, m, list(range(B)), prompts, split)
        assert not m.status().any(), name
        m.close()
        table.append((name, hl, ht))
    print("\n| configuration | logits hash | token hash |\n|---|---|---|")
    for name, hl, ht in table + [("CPU oracle (golden)", golden["logits_hash12"], golden["tokens_hash12"])]:
        print(f"| {name} | {hl} | {ht} |")
    assert {hl for _, hl, _ in table} == {golden["logits_hash12"]}
    assert {ht for _, _, ht in table} == {golden["tokens_hash12"]}
