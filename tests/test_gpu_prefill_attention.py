"""GPU parity of the tensor-core prefill attention (two sweeps over the keys:
row maxima, then 15-bit probabilities and the two int8 P·V limbs; DetLLM
blog, "DetLLM", footnote on 15-bit probabilities) against the CPU oracle:
chunked prefills whose query blocks start at unaligned positions, ragged
multi-sequence prefills, single-token prefills, and long prompts against the
per-token attention kernel. Tolerance 0."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

VOCAB = {"tiny": 1024, "qwen": 151936, "llama": 128256}


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deterministic_integer_only_gb300 as pkg
    pkg.lib()
    return torch


def _artifact(request, name):
    return request.getfixturevalue({"tiny": "tiny_artifact", "qwen": "qwen_artifact",
                                    "llama": "llama_artifact"}[name])


def _prefill(torch, m, sids, chunks):
    """One prefill call of several sequences; returns the logits rows."""
    dev = torch.device("cuda")
    cu = np.zeros(len(chunks) + 1, np.int64)
    cu[1:] = np.cumsum([len(c) for c in chunks])
    flat = torch.tensor(np.concatenate([np.asarray(c, np.int32) for c in chunks]),
                        dtype=torch.int32, device=dev)
    lg = torch.empty((len(chunks), m.vocab), dtype=torch.int32, device=dev)
    tok = torch.empty(len(chunks), dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        m.prefill(sids, flat, cu, lg, tok)
        out = lg.cpu().numpy(), tok.cpu().numpy()
    m.stream.synchronize()
    return out


@pytest.mark.parametrize("name", ["tiny", "qwen", "llama"])
@pytest.mark.parametrize("tc", [True, False])
def test_chunked_prefill_matches_oracle(torch_cuda, request, name, tc):
    import deterministic_integer_only_gb300 as pkg
    import oracle
    path = _artifact(request, name)
    prompt = synth.prompt_ids(3, 1, 300, VOCAB[name])
    bounds = np.cumsum([0, 37, 1, 100, 64, 98])
    m = pkg.Model(path, max_batch=2, max_ctx=320)
    m.set_tc_prefill(tc)
    om = oracle.Model(path)
    s = om.new_seq(320)
    for a, b in zip(bounds[:-1], bounds[1:]):
        lg, tok = _prefill(torch_cuda, m, [1], [prompt[a:b]])
        am, olg = s.feed(prompt[a:b])
        assert np.array_equal(lg[0], olg), (name, a, b)
        assert int(tok[0]) == am
    assert not m.status().any()
    m.close()


@pytest.mark.parametrize("name", ["tiny", "qwen"])
def test_ragged_multisequence_prefill_matches_oracle(torch_cuda, request, name):
    """Three sequences prefilled together twice: first prompts of lengths
    5, 70, 129, then continuations of 90, 1, 33 tokens from those positions."""
    import deterministic_integer_only_gb300 as pkg
    import oracle
    path = _artifact(request, name)
    V = VOCAB[name]
    first = [synth.prompt_ids(4, i, n, V) for i, n in enumerate((5, 70, 129))]
    second = [synth.prompt_ids(4, 10 + i, n, V) for i, n in enumerate((90, 1, 33))]
    sids = [2, 0, 3]
    m = pkg.Model(path, max_batch=4, max_ctx=256)
    lg1, _ = _prefill(torch_cuda, m, sids, first)
    lg2, tok2 = _prefill(torch_cuda, m, sids, second)
    om = oracle.Model(path)
    for b in range(3):
        s = om.new_seq(256)
        _, o1 = s.feed(first[b])
        am, o2 = s.feed(second[b])
        assert np.array_equal(lg1[b], o1), b
        assert np.array_equal(lg2[b], o2), b
        assert int(tok2[b]) == am
    m.close()


@pytest.mark.parametrize("name", ["qwen", "llama"])
def test_long_prefill_tc_equals_per_token(torch_cuda, request, name):
    """Two prompts of 1500 and 2100 tokens: the tensor-core attention gives
    the per-token kernel's logits, and the first prompt's last-position logits
    equal the oracle's."""
    import deterministic_integer_only_gb300 as pkg
    path = _artifact(request, name)
    V = VOCAB[name]
    prompts = [synth.prompt_ids(6, i, n, V) for i, n in enumerate((1500, 2100))]
    m = pkg.Model(path, max_batch=2, max_ctx=2112)
    out = {}
    for tc in (True, False):
        m.set_tc_prefill(tc)
        out[tc] = _prefill(torch_cuda, m, [0, 1], prompts)
        m.reset_seq(0)
        m.reset_seq(1)
    assert np.array_equal(out[True][0], out[False][0])
    assert np.array_equal(out[True][1], out[False][1])
    m.close()
    import oracle
    oracle.set_threads(oracle.max_threads())
    s = oracle.Model(path).new_seq(1500)
    am, olg = s.feed(prompts[0])
    assert np.array_equal(out[True][0][0], olg) and int(out[True][1][0]) == am
