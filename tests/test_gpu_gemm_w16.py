"""GPU parity of the exact int8 x int16 GEMM built from two int8 weight limbs
(BitExact LLM post, "Fix the arithmetic, not just the random seed": products
of split integer limbs combined in wider accumulators) against numpy int64,
every entry, including extreme operands and split-K grids."""
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


def test_split_limbs_exact(torch_cuda):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    W = np.concatenate([np.arange(-32768, 32768, dtype=np.int64),
                        np.random.default_rng(0).integers(-32768, 32768, 1000)]).astype(np.int16)
    hi, lo = pkg.detint_split_w16(torch.tensor(W, device="cuda"))
    hi, lo = hi.cpu().numpy().astype(np.int64), lo.cpu().numpy().astype(np.int64)
    assert np.array_equal(hi * 256 + lo, W.astype(np.int64))
    assert hi.min() >= -128 and hi.max() <= 127 and lo.min() >= 0 and lo.max() <= 255


def _run(torch, A, W):
    import deterministic_integer_only_gb300 as pkg
    hi, lo = pkg.detint_split_w16(torch.tensor(W, device="cuda"))
    C = torch.full((A.shape[0], W.shape[0]), 7, dtype=torch.int64, device="cuda")
    pkg.detint_gemm_w16(torch.tensor(A, device="cuda"), hi, lo, C)
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 17, 64), (33, 136, 144), (64, 520, 1040), (100, 256, 2064),
                                   (300, 384, 4096), (5, 2048, 8192), (129, 130, 272)])
def test_gemm_w16_exact(torch_cuda, M, N, K):
    rng = np.random.default_rng(M * 131 + N + K)
    A = rng.integers(-128, 128, (M, K)).astype(np.int8)
    W = rng.integers(-32768, 32768, (N, K)).astype(np.int16)
    got = _run(torch_cuda, A, W)
    assert np.array_equal(got, A.astype(np.int64) @ W.astype(np.int64).T)


def test_gemm_w16_extremes(torch_cuda):
    K = 8192
    A = np.full((3, K), -128, np.int8)
    A[1] = 127
    A[2, ::2] = 127
    W = np.full((4, K), -32768, np.int16)
    W[1] = 32767
    W[2, 1::2] = 32767
    W[3] = -1
    got = _run(torch_cuda, A, W)
    assert np.array_equal(got, A.astype(np.int64) @ W.astype(np.int64).T)


@pytest.mark.parametrize("M", [64, 512])
@pytest.mark.parametrize("N,K", [(2048, 2048), (16384, 2048), (2048, 8192)])
def test_gemm_w16_llama_shapes_sampled(torch_cuda, M, N, K):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    g = torch.Generator(device="cuda")
    g.manual_seed(M + N + K)
    a = torch.randint(-128, 128, (M, K), dtype=torch.int8, device="cuda", generator=g)
    w = torch.randint(-32768, 32768, (N, K), dtype=torch.int16, device="cuda", generator=g)
    hi, lo = pkg.detint_split_w16(w)
    c = pkg.detint_gemm_w16(a, hi, lo)
    rng = np.random.default_rng(M + N)
    rows, cols = rng.integers(0, M, 16), rng.integers(0, N, 64)
    Asub = a[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.int64)
    Wsub = w[torch.from_numpy(cols).cuda()].cpu().numpy().astype(np.int64)
    assert np.array_equal(c.cpu().numpy()[rows][:, cols], Asub @ Wsub.T)


def test_gemm_w16_rejects_bad_k(torch_cuda):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    a = torch.zeros((4, 20), dtype=torch.int8, device="cuda")
    hi = torch.zeros((4, 20), dtype=torch.int8, device="cuda")
    lo = torch.zeros((4, 20), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.DetintError) as e:
        pkg.detint_gemm_w16(a, hi, lo)
    assert e.value.code == 2
