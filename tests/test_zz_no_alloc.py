"""detint_argmax_noalloc: the tie-low argmax for callers that cannot allocate
device memory (inside an allocation-free stream capture, a host callback,
or an application that owns every allocation). Its partial results live in
a fixed device array, so this test checks it through the C ABI against the
token choice the decode entry points make with their own scratch, on two
calls in a row (the second must not see the first call's leftovers).

Collected last on purpose: a run that stops at the first failure has run
every other test before this one."""
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


def test_noalloc_argmax_matches_decode_token_choice(torch_cuda, tiny_artifact):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    dev = torch.device("cuda")
    m = pkg.Model(tiny_artifact, max_batch=4, max_ctx=64)
    prompts = [synth.prompt_ids(0, i, 9 + 3 * i, m.vocab) for i in range(4)]
    cu = np.zeros(5, np.int64)
    cu[1:] = np.cumsum([len(p) for p in prompts])
    flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
    logits = torch.empty((4, m.vocab), dtype=torch.int32, device=dev)
    tok = torch.empty(4, dtype=torch.int32, device=dev)
    out = torch.full((4,), -1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(m.stream):
        # call 1: the prefill's last-position logits of four sequences
        m.prefill([0, 1, 2, 3], flat, cu, logits, tok)
        pkg.detint_argmax_noalloc(logits, out, stream=m.stream)
        m.stream.synchronize()
        assert out.cpu().tolist() == tok.cpu().tolist()
        # call 2: a decode step's logits, fewer rows than call 1
        m.decode_step([0, 1, 2, 3], tok, logits, tok)
        out2 = torch.full((3,), -1, dtype=torch.int32, device=dev)
        pkg.detint_argmax_noalloc(logits[:3].contiguous(), out2, stream=m.stream)
        m.stream.synchronize()
        assert out2.cpu().tolist() == tok.cpu().tolist()[:3]
    # every row agrees with numpy's first-maximum rule as well
    lg = logits.cpu().numpy()
    assert out2.cpu().tolist() == [int(np.argmax(r)) for r in lg[:3]]
    m.close()


def test_noalloc_argmax_rejects_oversize(torch_cuda):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    x = torch.zeros((65, 8), dtype=torch.int32, device="cuda")
    out = torch.empty(65, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DetintError) as e:
        pkg.detint_argmax_noalloc(x, out)
    assert e.value.code == 2


def test_noalloc_argmax_across_chunks(torch_cuda):
    """Rows spanning many 4096-column chunks (151936 columns: 38 chunks, the
    last one partial) and the largest accepted shapes: equal maxima in
    different chunks go to the lower column, a row of INT32_MIN gives column
    0, and every row equals numpy's first maximum, on two calls in a row."""
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    rng = np.random.default_rng(77)
    imin, imax = np.iinfo(np.int32).min, np.iinfo(np.int32).max
    n = 151936
    x = rng.integers(imin, imax, (64, n), dtype=np.int64).astype(np.int32)
    x[0, 5 * 4096 + 17] = x[0, 20 * 4096 + 3] = imax            # tie in two chunks
    x[1, 30 * 4096 + 4000] = x[1, 30 * 4096 + 100] = imax        # tie inside one chunk
    x[1, 31 * 4096 + 1] = imax                                   # a later chunk ties too
    x[2, :] = imin                                               # all INT32_MIN
    x[3, n - 1] = imax                                           # the partial last chunk
    x[4, 0] = imax
    x[4, n - 1] = imax
    for call in range(2):
        xs = x if call == 0 else x[::-1].copy()
        t = torch.tensor(xs, device="cuda")
        out = torch.full((64,), -1, dtype=torch.int32, device="cuda")
        pkg.detint_argmax_noalloc(t, out)
        torch.cuda.synchronize()
        assert out.cpu().tolist() == [int(np.argmax(r)) for r in xs], call
    # the largest accepted sizes
    big = torch.tensor(rng.integers(-1000, 1000, (2, 1 << 20), dtype=np.int64).astype(np.int32), device="cuda")
    out = torch.empty(2, dtype=torch.int32, device="cuda")
    pkg.detint_argmax_noalloc(big, out)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [int(np.argmax(r)) for r in big.cpu().numpy()]
    full = torch.zeros((64, 64), dtype=torch.int32, device="cuda")
    full[:, 63] = 1
    out = torch.empty(64, dtype=torch.int32, device="cuda")
    pkg.detint_argmax_noalloc(full, out)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [63] * 64
