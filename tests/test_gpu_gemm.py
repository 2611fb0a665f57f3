"""GPU parity of detint_gemm_i8 (README, "Layout": int_gemm must return exact
results) against exact integer products computed on the CPU: numpy int64
brute force on small and ragged shapes, sampled entries at the Llama-shape
sweep sizes."""
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


def _run(torch, A, B):
    import deterministic_integer_only_gb300 as pkg
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = torch.empty((A.shape[0], B.shape[0]), dtype=torch.int32, device="cuda")
    pkg.detint_gemm_i8(a, b, c)
    torch.cuda.synchronize()
    return c.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (1, 17, 128), (3, 40, 256), (8, 4096, 1024),
                                   (9, 100, 192), (17, 1000, 320), (31, 333, 640),
                                   (32, 64, 8192), (33, 517, 640), (100, 250, 2048),
                                   (257, 129, 1024),
                                   # K a multiple of 16 only, ragged M/N tails of the 128 tiles
                                   (1, 1000, 80), (5, 33, 48), (40, 70, 16), (130, 200, 1040),
                                   (300, 389, 272)])
def test_gemm_small_exact(torch_cuda, M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    A = rng.integers(-127, 128, (M, K)).astype(np.int8)
    B = rng.integers(-127, 128, (N, K)).astype(np.int8)
    ref = (A.astype(np.int64) @ B.astype(np.int64).T)
    assert np.array_equal(_run(torch_cuda, A, B), ref)


def test_gemm_extremes(torch_cuda):
    K = 8192
    A = np.full((5, K), 127, np.int8)
    A[1] = -127
    B = np.full((70, K), -127, np.int8)
    B[3] = 127
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    got = _run(torch_cuda, A, B)
    assert np.array_equal(got, ref) and got.min() == -127 * 127 * K


@pytest.mark.parametrize("M", [1, 8, 64, 512, 4096])
@pytest.mark.parametrize("N,K", [(2048, 2048), (512, 2048), (3072, 2048), (16384, 2048),
                                 (2048, 8192), (128256, 2048)])
def test_gemm_llama_sweep_sampled(torch_cuda, M, N, K):
    torch = torch_cuda
    if M * N >= 4096 * 128256:
        pytest.skip("covered by the 512-row case of the same shape")
    g = torch.Generator(device="cuda")
    g.manual_seed(M + N + K)
    a = torch.randint(-127, 128, (M, K), dtype=torch.int8, device="cuda", generator=g)
    b = torch.randint(-127, 128, (N, K), dtype=torch.int8, device="cuda", generator=g)
    c = torch.empty((M, N), dtype=torch.int32, device="cuda")
    import deterministic_integer_only_gb300 as pkg
    pkg.detint_gemm_i8(a, b, c)
    rng = np.random.default_rng(M + N)
    rows = rng.integers(0, M, 16)
    cols = rng.integers(0, N, 64)
    A = a[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.int64)
    B = b[torch.from_numpy(cols).cuda()].cpu().numpy().astype(np.int64)
    got = c.cpu().numpy()[rows][:, cols]
    assert np.array_equal(got, A @ B.T)


@pytest.mark.parametrize("M,N,K", [(33, 136, 144), (50, 520, 1040), (64, 256, 2064), (65, 136, 1040),
                                   (100, 520, 2064), (200, 392, 784), (64, 130, 4112)])
def test_gemm_short_rows_and_split_k_exact(torch_cuda, M, N, K):
    """Every entry of the 64-row-tile and split-K paths (ragged M, N and a
    last k-tile that is partly past K) against numpy int64."""
    torch = torch_cuda
    import deterministic_integer_only_gb300 as pkg
    rng = np.random.default_rng(M * 7 + N + K)
    A = rng.integers(-127, 128, (M, K)).astype(np.int8)
    B = rng.integers(-127, 128, (N, K)).astype(np.int8)
    c = torch.full((M, N), 12345, dtype=torch.int32, device="cuda")
    pkg.detint_gemm_i8(torch.tensor(A, device="cuda"), torch.tensor(B, device="cuda"), c)
    assert np.array_equal(c.cpu().numpy(), A.astype(np.int64) @ B.astype(np.int64).T)


def test_gemm_rejects_bad_k(torch_cuda):
    import deterministic_integer_only_gb300 as pkg
    torch = torch_cuda
    a = torch.zeros((4, 20), dtype=torch.int8, device="cuda")
    b = torch.zeros((4, 20), dtype=torch.int8, device="cuda")
    c = torch.empty((4, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DetintError) as e:
        pkg.detint_gemm_i8(a, b, c)
    assert e.value.code == 2
