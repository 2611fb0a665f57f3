"""GPU parity of detint_sample (integer temperature, top-k, top-p and one
SplitMix64 draw; the BitExact LLM post's integer sampling rules, read as in
the arithmetic specification) against the CPU oracle, token for token: many
parameter sets, tie-heavy and extreme rows, the Qwen3-0.6B vocabulary, model
logits, more rows than one launch carries, and argument errors."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deterministic_integer_only_gb300 as pkg
    pkg.lib()
    return torch


def _rows(rng, kind, rows, n):
    if kind == "wide":
        return rng.integers(-(1 << 26), 1 << 26, (rows, n)).astype(np.int32)
    if kind == "ties":
        return (rng.integers(-6, 6, (rows, n)) << 16).astype(np.int32)
    if kind == "extreme":
        x = rng.integers(-(2 ** 31 - 1), 2 ** 31 - 1, (rows, n), dtype=np.int64).astype(np.int32)
        x[:, :3] = 2 ** 31 - 1
        return x
    return rng.integers(-(12 << 16), 12 << 16, (rows, n)).astype(np.int32)   # logit-like


PARAMS = [dict(inv_temp=65536), dict(inv_temp=0), dict(inv_temp=1 << 20), dict(inv_temp=30000, top_k=7),
          dict(top_k=1), dict(top_p=60000), dict(top_p=1), dict(top_k=50, top_p=30000),
          dict(inv_temp=90000, top_k=3, top_p=65000), dict(top_k=100000)]


@pytest.mark.parametrize("n", [1, 5, 1000, 4099])
@pytest.mark.parametrize("kind", ["logit", "ties", "wide", "extreme"])
def test_sample_matches_oracle(torch_cuda, n, kind):
    import deterministic_integer_only_gb300 as pkg
    import oracle
    torch = torch_cuda
    rng = np.random.default_rng(n * 7 + len(kind))
    for pi, prm in enumerate(PARAMS):
        x = _rows(rng, kind, 6, n)
        ps = [dict(prm, seed=1000 + pi, counter=r * 13 + 1) for r in range(6)]
        got = pkg.detint_sample(torch.tensor(x, device="cuda"), ps).cpu().numpy()
        want = [oracle.sample(x[r], ps[r].get("inv_temp", 65536), ps[r].get("top_k", 0),
                              ps[r].get("top_p", 65536), ps[r]["seed"], ps[r]["counter"]) for r in range(6)]
        assert got.tolist() == want, (kind, n, prm)


def test_sample_vocabulary_rows_and_many_counters(torch_cuda):
    """151936-wide rows (the Qwen3-0.6B vocabulary), 40 rows in one call (two
    launches), one seed with consecutive counters."""
    import deterministic_integer_only_gb300 as pkg
    import oracle
    torch = torch_cuda
    rng = np.random.default_rng(9)
    x = rng.integers(-(8 << 16), 8 << 16, (40, 151936)).astype(np.int32)
    x[3, 17] = x[3, 90000] = 30 << 16                      # a tied maximum
    ps = [dict(seed=5, counter=c, inv_temp=65536 + 500 * c, top_k=(0, 40, 1000)[c % 3],
               top_p=(65536, 58000)[c % 2]) for c in range(40)]
    got = pkg.detint_sample(torch.tensor(x, device="cuda"), ps).cpu().numpy()
    for r in range(40):
        p = ps[r]
        assert got[r] == oracle.sample(x[r], p["inv_temp"], p["top_k"], p["top_p"], 5, p["counter"]), r


def test_sample_model_logits(torch_cuda, tiny_artifact):
    """Logits of the tiny model's decode steps, sampled on the GPU and by the
    oracle with the same parameters."""
    import deterministic_integer_only_gb300 as pkg
    import oracle
    import synth
    torch = torch_cuda
    m = pkg.Model(tiny_artifact, max_batch=2, max_ctx=64)
    toks, rows = m.generate([synth.prompt_ids(0, 0, 16, 1024), synth.prompt_ids(0, 1, 9, 1024)], 6)
    m.close()
    lg = np.concatenate(rows, 0)
    p = dict(seed=77, inv_temp=70000, top_k=40, top_p=62000)
    ps = [dict(p, counter=c) for c in range(lg.shape[0])]
    got = pkg.detint_sample(torch.tensor(lg, device="cuda"), ps).cpu().numpy()
    want = [oracle.sample(lg[c], 70000, 40, 62000, 77, c) for c in range(lg.shape[0])]
    assert got.tolist() == want
    # top_k = 1 is the greedy token the decode itself chose
    greedy = pkg.detint_sample(torch.tensor(lg, device="cuda"), dict(top_k=1, seed=3)).cpu().numpy()
    assert greedy.tolist() == toks.T.reshape(-1).tolist()


def test_sample_rejects_bad_arguments(torch_cuda):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    x = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    for bad in (dict(inv_temp=-1), dict(inv_temp=(1 << 20) + 1), dict(top_p=0), dict(top_p=65537),
                dict(top_k=-2)):
        with pytest.raises(pkg.DetintError) as e:
            pkg.detint_sample(x, bad)
        assert e.value.code == 1


def test_sampled_generation_is_batch_invariant(torch_cuda, qwen_artifact):
    """Sampled tokens (temperature, top-k, top-p; counter = step) of a row are
    the same alone and inside a batch of three, and top_k = 1 sampling is the
    greedy decode (BitExact LLM post, "What the checks actually compare":
    sampled tokens compared under batching changes)."""
    import deterministic_integer_only_gb300 as pkg
    import synth
    prompts = [synth.prompt_ids(31, i, n, 151936) for i, n in enumerate((40, 7, 90))]
    prm = dict(seed=1234, inv_temp=80000, top_k=40, top_p=62000)
    m = pkg.Model(qwen_artifact, max_batch=4, max_ctx=256)
    t3, h3 = m.generate(prompts, 16, keep_logits="hash", sampling=prm)
    for sid in range(3):
        m.reset_seq(sid)
    t1, h1 = m.generate(prompts[:1], 16, keep_logits="hash", sampling=prm)
    assert np.array_equal(t3[0], t1[0]) and h3[0] == h1[0]
    for sid in range(3):
        m.reset_seq(sid)
    g, _ = m.generate(prompts, 8, keep_logits=False)
    for sid in range(3):
        m.reset_seq(sid)
    k1, _ = m.generate(prompts, 8, keep_logits=False, sampling=dict(top_k=1, seed=5))
    assert np.array_equal(g, k1)
    # at a high temperature the sampled stream leaves the greedy one
    for sid in range(3):
        m.reset_seq(sid)
    hot, _ = m.generate(prompts, 8, keep_logits=False, sampling=dict(seed=9, inv_temp=4000))
    assert not np.array_equal(hot, g)
    m.close()
