"""Host-side checks of the C ABI boundary (no GPU needed): the library
builds, loads, and exports every entry point include/detint.h declares; the
binding raises instead of falling back when the library is missing; kernel
sources contain no floating-point types, literals or runtime divisions."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "detint.h")
CSRC = os.path.join(ROOT, "deterministic_integer_only_gb300", "csrc")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(detint_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def built_lib():
    from deterministic_integer_only_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_library_exports_every_declared_symbol(built_lib):
    names = _declared()
    assert "detint_load" in names and "detint_gemm_i8" in names
    for n in names:
        assert hasattr(built_lib, n), n


def test_binding_symbol_list_matches_header():
    import deterministic_integer_only_gb300 as pkg
    assert sorted(pkg.SYMBOLS) == _declared()


def test_strerror_without_gpu(built_lib):
    built_lib.detint_strerror.restype = ctypes.c_char_p
    assert built_lib.detint_strerror(0) == b"ok"
    assert b"sha256" in built_lib.detint_strerror(6)


def test_load_rejects_missing_artifact_without_gpu(built_lib, tmp_path):
    h = ctypes.c_void_p()
    rc = built_lib.detint_load(str(tmp_path / "nope.detint").encode(), 1, 16, None, ctypes.byref(h))
    assert rc == 5 and not h.value


def test_load_rejects_corrupt_artifact_without_gpu(built_lib, tmp_path, tiny_artifact):
    # a flipped byte fails the SHA-256 check before any device work
    data = bytearray(open(tiny_artifact, "rb").read())
    data[1000] ^= 1
    p = tmp_path / "bad.detint"
    p.write_bytes(bytes(data))
    (tmp_path / "bad.detint.sha256").write_text(open(tiny_artifact + ".sha256").read())
    h = ctypes.c_void_p()
    rc = built_lib.detint_load(str(p).encode(), 1, 16, None, ctypes.byref(h))
    assert rc == 6 and not h.value
    os.remove(tmp_path / "bad.detint.sha256")
    rc = built_lib.detint_load(str(p).encode(), 1, 16, None, ctypes.byref(h))
    assert rc == 6


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from deterministic_integer_only_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.lib()


_FLOAT = re.compile(r"\b(float|double|half|__half|__nv_bfloat16|nv_bfloat16|float2|float4|"
                    r"__float2int_rn|__int2float_rn|__fdividef|sqrtf|expf|exp2f|logf|powf|"
                    r"__frcp_rn|rsqrtf)\b")
_FLOAT_LIT = re.compile(r"(?<![\w.])\d+\.\d*(?:[eE][-+]?\d+)?f?\b|(?<![\w.])\d+[eE][-+]?\d+")


def _kernel_sources():
    """Device code: every .cuh file (host launchers and the runtime are .cu)."""
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cuh")]


def _all_sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh"))]


def _code_only(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return re.sub(r'"(?:\\.|[^"\\])*"', '""', src)


def test_sources_have_no_floating_point():
    for path in _all_sources():
        code = _code_only(open(path).read())
        assert not _FLOAT.search(code), (path, _FLOAT.search(code).group(0))
        assert not _FLOAT_LIT.search(code), (path, _FLOAT_LIT.search(code).group(0))


def test_kernel_sources_divide_only_by_constants():
    # '/' or '%' must be followed by a literal, a constexpr name in CAPS/NTOK,
    # or a sizeof; a runtime divisor would go through CUDA's division sequence
    ok = re.compile(r"^\s*(\(?\d+|[A-Z_][A-Z0-9_]*\b|sizeof)")
    for path in _kernel_sources():
        code = _code_only(open(path).read())
        for m in re.finditer(r"(?<![/*])([/%])(?![/*=])", code):
            rest = code[m.end():m.end() + 40]
            line = code[:m.start()].count("\n") + 1
            assert ok.match(rest), f"{os.path.basename(path)}:{line}: divisor {rest.split()[0]!r}"
