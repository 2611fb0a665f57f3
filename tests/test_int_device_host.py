"""The scalar integer routines of the kernels' device header, built for the
host, against the oracle on the same inputs: the rounding shift, floor square
root, 15-bit dyadic scales, the cubic exp2 in Q15, the SwiGLU channel
(DetLLM blog, section "DetLLM": fixed rounding rules, integer exp and
activation) and the exact mode's 128-bit requantisation (BitExact LLM post,
"Three execution paths"). The GPU parity tests cover these routines inside the kernels;
this catches a change to the header without a GPU."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def host_run(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("intdev")
    exe = str(d / "host_int_device")
    r = subprocess.run([nvcc, "-O2", "-x", "cu", os.path.join(HERE, "host_int_device.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    rng = np.random.default_rng(20250601)
    n = 200_000
    inputs = {}
    # rounding shift: |x| < 2^62, s in [0, 40], with exact ties
    x = rng.integers(-(1 << 62), 1 << 62, n, dtype=np.int64)
    s = rng.integers(0, 41, n).astype(np.int32)
    ties = (np.arange(1, 2001, dtype=np.int64) * 2 + 1) << 9      # odd multiples of 2^9
    x[:4000] = np.concatenate([ties, -ties])
    s[:4000] = 10
    inputs["rshr_x"], inputs["rshr_s"] = x, s
    # floor square root: random below 2^62 and squares +-1
    q = rng.integers(0, 1 << 62, n, dtype=np.uint64)
    rt = rng.integers(1, 1 << 31, 20000, dtype=np.uint64)
    q[:60000] = np.concatenate([rt * rt, rt * rt - np.uint64(1), rt * rt + np.uint64(1)])
    inputs["isqrt_x"] = q
    # the single-thread square root: every bit length (log-uniform), squares
    # +-1 of every root length, all n below 2^16 and the top of the range
    bl = rng.integers(1, 63, n).astype(np.uint64)
    qf = (rng.integers(0, 1 << 62, n, dtype=np.uint64) << np.uint64(2)) >> (np.uint64(64) - bl)
    rb = rng.integers(1, 32, 30000).astype(np.uint64)
    rf = (rng.integers(0, 1 << 31, 30000, dtype=np.uint64) >> (np.uint64(31) - rb)) | (np.uint64(1) << (rb - np.uint64(1)))
    sq = rf * rf
    qf[:90000] = np.concatenate([sq, sq - np.uint64(1), sq + np.uint64(1)])
    qf[90000:90000 + (1 << 16)] = np.arange(1 << 16, dtype=np.uint64)
    qf[-3:] = [(1 << 62) - 1, 1 << 61, (1 << 60) - 1]
    inputs["isqrtf_x"] = qf
    # dyadic scales over the kernels' ranges (N, D below 2^40, |k| <= 39)
    ln = rng.integers(1, 41, n)
    ld = np.clip(ln - 14 + rng.integers(-39, 40, n), 1, 40)
    inputs["dyadic_n"] = (rng.integers(0, 1 << 62, n, dtype=np.uint64) >> (64 - ln).astype(np.uint64)) | (
        np.uint64(1) << (ln - 1).astype(np.uint64))
    inputs["dyadic_d"] = (rng.integers(0, 1 << 62, n, dtype=np.uint64) >> (64 - ld).astype(np.uint64)) | (
        np.uint64(1) << (ld - 1).astype(np.uint64))
    # exp2 exponent: every delta from -25 * 1024 to 0
    inputs["exp2q_d"] = np.arange(-25 * 1024, 1, dtype=np.int64)
    # SwiGLU on saturated Q12 gate/up values, dense near zero
    g = rng.integers(-(1 << 24), (1 << 24) + 1, n).astype(np.int32)
    u = rng.integers(-(1 << 24), (1 << 24) + 1, n).astype(np.int32)
    g[:50001] = np.arange(-25000, 25001, dtype=np.int32)
    g[50001:50005] = [1 << 24, -(1 << 24), 0, 1]
    u[50001:50005] = [1 << 24, 1 << 24, -(1 << 24), -(1 << 24)]
    inputs["swiglu_g"], inputs["swiglu_u"] = g, u
    # exact-mode requantisation: int64 accumulators of 16-bit weights
    acc = rng.integers(-(1 << 35), 1 << 35, n, dtype=np.int64)
    acc[:1000] = rng.integers(-4096, 4096, 1000)
    mt = rng.integers(1 << 14, (1 << 15) + 1, n).astype(np.int32)
    mc = rng.integers(1 << 14, 1 << 15, n).astype(np.int32)
    kt = rng.integers(-2, 40, n).astype(np.int32)
    inputs["mul128_acc"] = acc
    inputs["mul128_m"] = (mt.astype(np.int64) * mc.astype(np.int64)).astype(np.uint64)
    inputs["mul128_s"] = (kt + 30 - 16).astype(np.int32)
    inputs["_mt"], inputs["_mc"], inputs["_kt"] = mt, mc, kt
    # planted exact ties of both signs (acc * M an odd multiple of 2^(s-1))
    # and shifts 60..100 whose results fit int64
    xa, xm, xs = [], [], []
    for i in range(4000):
        s_ = int(rng.integers(2, 64))
        j = int(rng.integers(0, min(31, s_ - 1) + 1))       # M = 2^j
        k = 2 * int(rng.integers(0, 1 << 12)) + 1            # odd
        a_ = k << (s_ - 1 - j)
        if abs(a_) >= 1 << 36:
            continue
        xa.append(a_ if i % 2 else -a_); xm.append(1 << j); xs.append(s_)
    for i in range(4000):
        s_ = int(rng.integers(60, 101))
        a_ = int(rng.integers(-(1 << 35), 1 << 35))
        m_ = int(rng.integers(1, 1 << 31))
        xa.append(a_); xm.append(m_); xs.append(s_)
    inputs["mul128x_acc"] = np.array(xa, np.int64)
    inputs["mul128x_m"] = np.array(xm, np.uint64)
    inputs["mul128x_s"] = np.array(xs, np.int32)
    for k, v in inputs.items():
        if not k.startswith("_"):
            v.tofile(str(d / f"{k}.bin"))
    r = subprocess.run([exe, str(d)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def out(name, dt):
        return np.fromfile(str(d / f"{name}.bin"), dtype=dt)

    return inputs, out


def test_rshr(host_run):
    inp, out = host_run
    np.testing.assert_array_equal(out("rshr_out", np.int64), oracle.rshr(inp["rshr_x"], inp["rshr_s"]))


def test_isqrt(host_run):
    inp, out = host_run
    np.testing.assert_array_equal(out("isqrt_out", np.uint64), oracle.isqrt(inp["isqrt_x"]))


def test_isqrt_fast(host_run):
    """The single-thread Newton-Raphson square root equals the oracle's."""
    inp, out = host_run
    np.testing.assert_array_equal(out("isqrtf_out", np.uint64), oracle.isqrt(inp["isqrtf_x"]))


def test_dyadic(host_run):
    inp, out = host_run
    m, k = oracle.dyadic(inp["dyadic_n"].astype(np.int64), inp["dyadic_d"].astype(np.int64))
    np.testing.assert_array_equal(out("dyadic_m", np.int32), m)
    np.testing.assert_array_equal(out("dyadic_k", np.int32), k)


def test_dyadic_fast(host_run):
    """The single-thread dyadic (Newton-Raphson division) equals the oracle's."""
    inp, out = host_run
    m, k = oracle.dyadic(inp["dyadic_n"].astype(np.int64), inp["dyadic_d"].astype(np.int64))
    np.testing.assert_array_equal(out("dyadicf_m", np.int32), m)
    np.testing.assert_array_equal(out("dyadicf_k", np.int32), k)


def test_exp2q(host_run):
    inp, out = host_run
    np.testing.assert_array_equal(out("exp2q_out", np.int64), oracle.exp2q(inp["exp2q_d"]))


def test_swiglu(host_run):
    inp, out = host_run
    np.testing.assert_array_equal(out("swiglu_out", np.int32), oracle.swiglu(inp["swiglu_g"], inp["swiglu_u"]))


def test_requant_mul128(host_run):
    inp, out = host_run
    want = oracle.requant_wide(inp["mul128_acc"], inp["_mt"], inp["_kt"], inp["_mc"], 16)
    np.testing.assert_array_equal(out("mul128_out", np.int64), want)


def test_mul128_ties_and_wide_shifts(host_run):
    """rshr_mul128 against the exact definition (Python integers): planted
    ties of both signs round toward +infinity, and shifts of 60..100."""
    inp, out = host_run
    got = out("mul128x_out", np.int64)
    for a_, m_, s_, g_ in zip(inp["mul128x_acc"].tolist(), inp["mul128x_m"].tolist(),
                              inp["mul128x_s"].tolist(), got.tolist()):
        assert g_ == (a_ * m_ + (1 << (s_ - 1))) >> s_, (a_, m_, s_)
