"""Scheduler invariance on the GPU (BitExact LLM post, "What the checks
actually compare": mixed requests, chunked prefill, shared prefixes and
preemption leave the outputs unchanged): sequences forked from a shared
prefix (KV blocks shared by reference count), a batch of forks decoding
together, preemption with recomputation, and block-pool exhaustion and
reuse. Every comparison is bit-exact, and every forked, batched or
recomputed row is also compared with the CPU oracle fed the same token
list (its prefill logits, greedy tokens and logits chain hash)."""
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


def _prefill(torch, m, sids, chunks):
    dev = torch.device("cuda")
    cu = np.zeros(len(chunks) + 1, np.int64)
    cu[1:] = np.cumsum([len(c) for c in chunks])
    flat = torch.tensor(np.concatenate([np.asarray(c, np.int32) for c in chunks]), dtype=torch.int32,
                        device=dev)
    lg = torch.empty((len(chunks), m.vocab), dtype=torch.int32, device=dev)
    tok = torch.empty(len(chunks), dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        m.prefill(sids, flat, cu, lg, tok)
    m.stream.synchronize()
    return lg.cpu().numpy(), tok


def _oracle(path, tokens, steps):
    """The oracle's last-position logits for the token list, then `steps`
    greedy tokens and the chain hash of their logits, as _decode reports."""
    import hashlib
    import oracle
    oracle.set_threads(oracle.max_threads())
    s = oracle.Model(path).new_seq(len(tokens) + steps + 1)
    am, lg0 = s.feed(np.asarray(tokens, np.int32))
    toks, h = [], b"\0" * 32
    for _ in range(steps):
        am, lg = s.feed([am])
        toks.append(am)
        h = hashlib.sha256(h + lg.astype("<i4").tobytes()).digest()
    return lg0, np.array(toks, np.int32), h


def _decode(torch, m, sids, tok, steps):
    """greedy steps; returns (tokens [steps][B], logits hash per row)"""
    import hashlib
    dev = torch.device("cuda")
    lg = torch.empty((len(sids), m.vocab), dtype=torch.int32, device=dev)
    out, hs = [], [b"\0" * 32] * len(sids)
    with torch.cuda.stream(m.stream):
        for _ in range(steps):
            m.decode_step(sids, tok, lg, tok)
            x = lg.cpu().numpy()
            out.append(tok.cpu().numpy().copy())
            hs = [hashlib.sha256(hs[b] + x[b].astype("<i4").tobytes()).digest() for b in range(len(sids))]
    return np.array(out), hs


@pytest.mark.parametrize("name,n_shared", [("tiny", 100), ("tiny", 128), ("qwen", 77), ("llama", 64)])
def test_fork_equals_fresh_prefill(torch_cuda, request, name, n_shared):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    path = request.getfixturevalue({"tiny": "tiny_artifact", "qwen": "qwen_artifact",
                                    "llama": "llama_artifact"}[name])
    V = {"tiny": 1024, "qwen": 151936, "llama": 128256}[name]
    base = synth.prompt_ids(21, 0, 150, V)
    tail = synth.prompt_ids(21, 1, 23, V)
    m = pkg.Model(path, max_batch=4, max_ctx=256)
    _prefill(torch, m, [0], [base])
    m.fork_seq(0, 1, n_shared)
    assert m.seq_len(1) == n_shared
    lg_f, tok_f = _prefill(torch, m, [1], [tail])
    toks_f, h_f = _decode(torch, m, [1], tok_f, 10)
    # the source continues unaffected
    lg_s, tok_s = _prefill(torch, m, [0], [tail[:5]])
    toks_s, h_s = _decode(torch, m, [0], tok_s, 6)
    # fresh sequences with the same token lists
    m.reset_seq(2)
    lg_r, tok_r = _prefill(torch, m, [2], [np.concatenate([base[:n_shared], tail])])
    toks_r, h_r = _decode(torch, m, [2], tok_r, 10)
    assert np.array_equal(lg_f, lg_r) and np.array_equal(toks_f, toks_r) and h_f == h_r
    m.reset_seq(3)
    lg_r2, tok_r2 = _prefill(torch, m, [3], [np.concatenate([base, tail[:5]])])
    toks_r2, h_r2 = _decode(torch, m, [3], tok_r2, 6)
    assert np.array_equal(lg_s, lg_r2) and np.array_equal(toks_s, toks_r2) and h_s == h_r2
    m.close()
    # both rows against the oracle
    o_lg, o_t, o_h = _oracle(path, np.concatenate([base[:n_shared], tail]), 10)
    assert np.array_equal(lg_f[0], o_lg) and np.array_equal(toks_f[:, 0], o_t) and h_f[0] == o_h
    o_lg, o_t, o_h = _oracle(path, np.concatenate([base, tail[:5]]), 6)
    assert np.array_equal(lg_s[0], o_lg) and np.array_equal(toks_s[:, 0], o_t) and h_s[0] == o_h


def test_batch_of_forks_decodes_like_solo_runs(torch_cuda, qwen_artifact):
    """Four sequences forked from one 130-token prefix at different points,
    each extended by its own tokens, then decoded together as one batch:
    every row equals that sequence's solo run."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    V = 151936
    base = synth.prompt_ids(22, 0, 130, V)
    cuts = (130, 64, 91, 1)
    tails = [synth.prompt_ids(22, 10 + i, 7 + 5 * i, V) for i in range(4)]
    m = pkg.Model(qwen_artifact, max_batch=5, max_ctx=256)
    _prefill(torch, m, [4], [base])
    for i, c in enumerate(cuts):
        m.fork_seq(4, i, c)
    _, tok = _prefill(torch, m, [0, 1, 2, 3], tails)
    toks_b, h_b = _decode(torch, m, [0, 1, 2, 3], tok, 12)
    for i, c in enumerate(cuts):
        m.reset_seq(i)
        _, t1 = _prefill(torch, m, [i], [np.concatenate([base[:c], tails[i]])])
        toks_1, h_1 = _decode(torch, m, [i], t1, 12)
        assert np.array_equal(toks_1[:, 0], toks_b[:, i]) and h_1[0] == h_b[i], i
    m.close()
    for i, c in enumerate(cuts):
        _, o_t, o_h = _oracle(qwen_artifact, np.concatenate([base[:c], tails[i]]), 12)
        assert np.array_equal(toks_b[:, i], o_t) and h_b[i] == o_h, i


def test_preempt_and_recompute(torch_cuda, tiny_artifact):
    """A sequence preempted mid-generation (its KV blocks freed) and later
    recomputed from its token history continues exactly as if uninterrupted."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    prompts = [synth.prompt_ids(23, i, n, 1024) for i, n in enumerate((40, 90))]
    m = pkg.Model(tiny_artifact, max_batch=2, max_ctx=256)
    _, tok = _prefill(torch, m, [0, 1], prompts)
    full, _ = _decode(torch, m, [0, 1], tok.clone(), 30)
    m.reset_seq(0)
    m.reset_seq(1)
    _, tok = _prefill(torch, m, [0, 1], prompts)
    g0 = tok.cpu().numpy().copy()       # the prefill's token, fed by the first step
    first, _ = _decode(torch, m, [0, 1], tok, 12)
    m.reset_seq(1)                      # preempt sequence 1; sequence 0 keeps running
    part0, _ = _decode(torch, m, [0], tok[:1].clone(), 5)
    # recompute: the prompt plus every token fed so far; the prefill returns
    # the token that was next
    _, t1 = _prefill(torch, m, [1], [np.concatenate([prompts[1], g0[1:2], first[:-1, 1]])])
    assert int(t1[0].item()) == int(first[-1, 1])
    rest1, _ = _decode(torch, m, [1], t1, 18)
    assert np.array_equal(np.concatenate([first[:, 1], rest1[:, 0]]), full[:, 1])
    assert np.array_equal(np.concatenate([first[:, 0], part0[:, 0]]), full[:17, 0])
    m.close()
    # the uninterrupted runs (which the preempted and recomputed ones equal) against the oracle
    for b in range(2):
        _, o_t, _ = _oracle(tiny_artifact, prompts[b], 30)
        assert np.array_equal(full[:, b], o_t), b


def test_fork_arguments_and_block_reuse(torch_cuda, tiny_artifact):
    """Forks that share whole blocks or copy a partial one, a non-empty
    destination refused, and freed blocks reused by later sequences."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    m = pkg.Model(tiny_artifact, max_batch=2, max_ctx=128)        # 4 blocks in the pool
    p = synth.prompt_ids(24, 0, 128, 1024)
    _prefill(torch, m, [0], [p])
    m.fork_seq(0, 1, 128)                                          # shares both blocks
    m.reset_seq(1)
    m.fork_seq(0, 1, 100)                                          # one shared, one copied
    with pytest.raises(pkg.DetintError) as e:
        m.fork_seq(0, 1, 10)                                       # dst not empty
    assert e.value.code == 9
    m.reset_seq(0)
    m.reset_seq(1)
    lg1, _ = _prefill(torch, m, [1], [p[:100]])
    m.reset_seq(1)
    lg2, _ = _prefill(torch, m, [0], [p[:100]])
    assert np.array_equal(lg1, lg2)
    m.close()
