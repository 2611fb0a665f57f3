"""Writes oracle_tiny_seed0.json: the CPU oracle's token stream and chain
hashes for the tiny model (seed 0, 16-token seeded prompt, 16 greedy steps),
oracle_tiny_w16_seed0.json: the same for the tiny model's wide-weight
(exact-mode) artifact, and oracle_qwen06b_demo.json: the same for the
Qwen3-0.6B-shaped model on the pages' demo workload (64-token seeded prompt,
512 greedy steps; DetLLM README, "Demo").

With --full it also writes the full-size fixtures (minutes of oracle time):
oracle_qwen06b_split2048.json (a 2048-token seeded prompt then 512 greedy
steps, the split-prefill workload; DetLLM README, "Demo": split prefill gives
the same hash), oracle_qwen06b_prefill4096.json (the last-position logits of a
4096-token prompt; DetLLM blog, footnote on the zero-tolerance suite: prefill
against token-by-token decoding up to a 4k context) and
oracle_llama1b_ctx1024.json (two of the 32 batch-32 Llama-shaped sequences,
1024-token contexts and 16 greedy steps each).

It calls only the oracle and the seeded input generator; no value in the
fixture comes from the CUDA path. Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402
import synth   # noqa: E402


def run(shape, seed, prompt_len, steps, max_ctx, wide=False):
    path = synth.ensure_artifact(shape, seed, wide=wide)
    oracle.set_threads(oracle.max_threads())
    m = oracle.Model(path)
    ids = synth.prompt_ids(seed, 0, prompt_len, m.vocab)
    s = m.new_seq(max_ctx)
    am, lg = s.feed(ids)
    h, toks = oracle.chain_hash([lg]), [am]
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        h = oracle.chain_hash([lg], h)
        toks.append(am)
    return {
        "what": f"CPU oracle, {shape} model{' (16-bit weights)' if wide else ''}, seed {seed}, "
                f"prompt index 0, greedy",
        "seed": seed, "prompt_len": prompt_len, "steps": steps,
        "artifact_sha256": open(path + ".sha256").read().strip(),
        "tokens": toks,
        "logits_hash12": h.hex()[:12],
        "tokens_hash12": oracle.chain_hash([np.array([t], np.int32) for t in toks]).hex()[:12],
    }


def run_rows(shape, seed, pseed, index, prompt_len, steps, max_ctx):
    """Tokens and chain hashes of the artifact (shape, seed) on the seeded
    prompt (pseed, index) followed by greedy steps; the oracle feeds the
    prompt token by token."""
    path = synth.ensure_artifact(shape, seed)
    oracle.set_threads(oracle.max_threads())
    m = oracle.Model(path)
    ids = synth.prompt_ids(pseed, index, prompt_len, m.vocab)
    s = m.new_seq(max_ctx)
    am, lg = s.feed(ids)
    last = lg.copy()
    h, toks = oracle.chain_hash([lg]), [am]
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        h = oracle.chain_hash([lg], h)
        toks.append(am)
    return {
        "seed": seed, "prompt_seed": pseed, "index": index, "prompt_len": prompt_len,
        "steps": steps, "artifact_sha256": open(path + ".sha256").read().strip(),
        "tokens": toks,
        "prefill_logits_hash12": oracle.chain_hash([last]).hex()[:12],
        "logits_hash12": h.hex()[:12],
        "tokens_hash12": oracle.chain_hash([np.array([t], np.int32) for t in toks]).hex()[:12],
    }


def write_full(here):
    out = run_rows("qwen3-0.6b", 0, 0, 7, 2048, 512, 2048 + 512)
    out["what"] = ("CPU oracle, qwen3-0.6b model, seed 0, prompt index 7 (2048 tokens), "
                   "512 greedy steps; step 0 is the prompt's last-position logits")
    with open(os.path.join(here, "oracle_qwen06b_split2048.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print({k: v for k, v in out.items() if k != "tokens"})
    out = run_rows("qwen3-0.6b", 0, 0, 8, 4096, 1, 4096)
    out["what"] = ("CPU oracle, qwen3-0.6b model, seed 0, prompt index 8 (4096 tokens): "
                   "the last position's logits hash and argmax")
    with open(os.path.join(here, "oracle_qwen06b_prefill4096.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print({k: v for k, v in out.items() if k != "tokens"})
    rows = {}
    for b in (0, 17):
        rows[str(b)] = run_rows("llama-1b", 0, 9, b, 1024, 16, 1024 + 16)
        print(b, {k: v for k, v in rows[str(b)].items() if k != "tokens"})
    with open(os.path.join(here, "oracle_llama1b_ctx1024.json"), "w") as f:
        json.dump({"what": "CPU oracle, llama-1b model, seed 0, prompt seed 9, indices 0 and 17 "
                           "(1024 tokens each), 16 greedy steps each", "rows": rows}, f, indent=1)
        f.write("\n")


def write_wide(here):
    wide = run("tiny", 0, 16, 16, 64, wide=True)
    with open(os.path.join(here, "oracle_tiny_w16_seed0.json"), "w") as f:
        json.dump(wide, f, indent=1)
        f.write("\n")
    print({k: v for k, v in wide.items() if k != "tokens"})


def main():
    here = os.path.dirname(os.path.abspath(__file__))
    if "--full" in sys.argv:
        write_full(here)
        return
    write_wide(here)
    if "--wide-only" in sys.argv:
        return
    demo = run("qwen3-0.6b", 0, 64, 512, 640)
    with open(os.path.join(here, "oracle_qwen06b_demo.json"), "w") as f:
        json.dump(demo, f, indent=1)
        f.write("\n")
    print({k: v for k, v in demo.items() if k != "tokens"})
    seed, prompt_len, steps = 0, 16, 16
    path = synth.ensure_artifact("tiny", seed)
    m = oracle.Model(path)
    ids = synth.prompt_ids(seed, 0, prompt_len, m.vocab)
    s = m.new_seq(64)
    am, lg = s.feed(ids)
    rows, toks = [lg], [am]
    for _ in range(steps - 1):
        am, lg = s.feed([toks[-1]])
        rows.append(lg)
        toks.append(am)
    out = {
        "what": "CPU oracle, tiny model, seed 0, prompt index 0, greedy",
        "seed": seed, "prompt_len": prompt_len, "steps": steps,
        "artifact_sha256": open(path + ".sha256").read().strip(),
        "tokens": toks,
        "logits_hash12": oracle.chain_hash(rows).hex()[:12],
        "tokens_hash12": oracle.chain_hash([np.array([t], np.int32) for t in toks]).hex()[:12],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_seed0.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(out)


if __name__ == "__main__":
    main()
