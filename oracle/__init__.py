"""ctypes front end of the detint CPU oracle (test infrastructure only).

The oracle (detint_oracle.c, plain scalar int64 C) defines the expected bits
of the integer-only forward pass. Only the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the product path never imports it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "detint_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over output channels only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-shared", "-fPIC", "-Wall",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(C.POINTER(t))


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        i64, i32, u64 = C.c_int64, C.c_int32, C.c_uint64
        L.or_rshr.restype = i64; L.or_rshr.argtypes = [i64, C.c_int]
        L.or_isqrt.restype = u64; L.or_isqrt.argtypes = [u64]
        L.or_exp2q.restype = i64; L.or_exp2q.argtypes = [i64]
        L.or_requant.restype = i64; L.or_requant.argtypes = [i64, i32, i32, i32, C.c_int]
        L.or_swiglu.restype = i32; L.or_swiglu.argtypes = [i32, i32]
        L.or_last_error.restype = C.c_char_p
        L.or_model_load.restype = C.c_void_p
        L.or_model_load.argtypes = [C.c_char_p, C.POINTER(C.c_int)]
        L.or_model_free.argtypes = [C.c_void_p]
        L.or_model_info.argtypes = [C.c_void_p, C.POINTER(i32)]
        L.or_seq_new.restype = C.c_void_p; L.or_seq_new.argtypes = [C.c_void_p, C.c_int]
        L.or_seq_free.argtypes = [C.c_void_p]
        L.or_seq_len.argtypes = [C.c_void_p]
        L.or_seq_feed.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.POINTER(i32),
                                  C.POINTER(i32), C.POINTER(i32)]
        L.or_splitmix64.restype = u64; L.or_splitmix64.argtypes = [u64, u64]
        L.or_sample.restype = C.c_int
        L.or_sample.argtypes = [C.POINTER(i32), C.c_int, i32, i32, i32, u64, u64]
        L.or_sample_set.restype = C.c_int
        L.or_sample_set.argtypes = [C.POINTER(i32), C.c_int, i32, i32, i32, C.POINTER(C.c_char),
                                    C.POINTER(i64), C.POINTER(i64)]
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def check():
    L = lib()
    if L.or_error_count():
        msg = L.or_last_error().decode()
        L.or_clear_error()
        raise OracleError(msg)


def set_threads(n: int):
    lib().or_set_threads(int(n))


def max_threads() -> int:
    return int(lib().or_max_threads())


# ---------------------------------------------------------------- primitives
def rshr(x, s):
    x = np.ascontiguousarray(x, dtype=np.int64).ravel()
    s = np.broadcast_to(np.asarray(s, dtype=np.int32), x.shape).copy()
    out = np.empty_like(x)
    lib().or_rshr_vec(_p(x, C.c_int64), _p(s, C.c_int32), _p(out, C.c_int64), C.c_int(x.size))
    check()
    return out


def isqrt(x):
    x = np.ascontiguousarray(x, dtype=np.uint64).ravel()
    out = np.empty_like(x)
    lib().or_isqrt_vec(_p(x, C.c_uint64), _p(out, C.c_uint64), C.c_int(x.size))
    check()
    return out


def dyadic(N, D):
    N = np.ascontiguousarray(N, dtype=np.int64).ravel()
    D = np.broadcast_to(np.asarray(D, dtype=np.int64), N.shape).copy()
    m = np.empty(N.size, np.int32)
    k = np.empty(N.size, np.int32)
    lib().or_dyadic_vec(_p(N, C.c_int64), _p(D, C.c_int64), _p(m, C.c_int32), _p(k, C.c_int32),
                        C.c_int(N.size))
    check()
    return m, k


def exp2q(delta):
    d = np.ascontiguousarray(delta, dtype=np.int64).ravel()
    out = np.empty_like(d)
    lib().or_exp2q_vec(_p(d, C.c_int64), _p(out, C.c_int64), C.c_int(d.size))
    check()
    return out


def swiglu(g, u):
    g = np.ascontiguousarray(g, dtype=np.int32).ravel()
    u = np.ascontiguousarray(u, dtype=np.int32).ravel()
    out = np.empty_like(g)
    lib().or_swiglu_vec(_p(g, C.c_int32), _p(u, C.c_int32), _p(out, C.c_int32), C.c_int(g.size))
    check()
    return out


def requant(acc, mt, kt, mc, f_out):
    acc = np.ascontiguousarray(acc, dtype=np.int64).ravel()
    n = acc.size
    mt = np.broadcast_to(np.asarray(mt, np.int32), (n,)).copy()
    kt = np.broadcast_to(np.asarray(kt, np.int32), (n,)).copy()
    mc = np.broadcast_to(np.asarray(mc, np.int32), (n,)).copy()
    out = np.empty(n, np.int64)
    lib().or_requant_vec(_p(acc, C.c_int64), _p(mt, C.c_int32), _p(kt, C.c_int32),
                         _p(mc, C.c_int32), C.c_int(f_out), _p(out, C.c_int64), C.c_int(n))
    check()
    return out


def requant_wide(acc, mt, kt, mc, f_out):
    """Requantisation of an int64 accumulator of 16-bit weights (scale
    m_c / 2^30), one exact 128-bit product and one rounding shift."""
    acc = np.ascontiguousarray(acc, dtype=np.int64).ravel()
    n = acc.size
    mt = np.broadcast_to(np.asarray(mt, np.int32), (n,)).copy()
    kt = np.broadcast_to(np.asarray(kt, np.int32), (n,)).copy()
    mc = np.broadcast_to(np.asarray(mc, np.int32), (n,)).copy()
    out = np.empty(n, np.int64)
    lib().or_requant_wide_vec(_p(acc, C.c_int64), _p(mt, C.c_int32), _p(kt, C.c_int32),
                              _p(mc, C.c_int32), C.c_int(f_out), _p(out, C.c_int64), C.c_int(n))
    check()
    return out


def actquant(x, F):
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.int32)
    rows, n = x.shape
    q = np.empty((rows, n), np.int8)
    mt = np.empty(rows, np.int32)
    kt = np.empty(rows, np.int32)
    lib().or_actquant_rows(_p(x, C.c_int32), C.c_int(rows), C.c_int(n), C.c_int(F),
                           _p(q, C.c_int8), _p(mt, C.c_int32), _p(kt, C.c_int32))
    check()
    return q, mt, kt


def normquant(x, gamma, eps):
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.int32)
    gamma = np.ascontiguousarray(gamma, dtype=np.int16)
    rows, n = x.shape
    q = np.empty((rows, n), np.int8)
    mt = np.empty(rows, np.int32)
    kt = np.empty(rows, np.int32)
    lib().or_normquant_rows(_p(x, C.c_int32), C.c_int(rows), C.c_int(n), _p(gamma, C.c_int16),
                            C.c_int64(eps), _p(q, C.c_int8), _p(mt, C.c_int32), _p(kt, C.c_int32))
    check()
    return q, mt, kt


def qknorm(x, gamma, eps):
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.int32)
    gamma = np.ascontiguousarray(gamma, dtype=np.int16)
    rows, n = x.shape
    y = np.empty((rows, n), np.int32)
    lib().or_qknorm_rows(_p(x, C.c_int32), C.c_int(rows), C.c_int(n), _p(gamma, C.c_int16),
                         C.c_int64(eps), _p(y, C.c_int32))
    check()
    return y


def rope(y, cos_row, sin_row):
    y = np.ascontiguousarray(y, dtype=np.int32).copy()
    c = np.ascontiguousarray(cos_row, dtype=np.int16)
    s = np.ascontiguousarray(sin_row, dtype=np.int16)
    lib().or_rope(_p(y, C.c_int32), C.c_int(y.size), _p(c, C.c_int16), _p(s, C.c_int16))
    check()
    return y


def gemm_i8(A, B):
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, K = A.shape
    N = B.shape[0]
    Cm = np.empty((M, N), np.int32)
    lib().or_gemm_i8(_p(A, C.c_int8), _p(B, C.c_int8), _p(Cm, C.c_int32), C.c_int(M), C.c_int(N),
                     C.c_int(K))
    check()
    return Cm


def attention_row(q8, mq, kq, K8, V8, kvp):
    q8 = np.ascontiguousarray(q8, np.int8)
    K8 = np.ascontiguousarray(K8, np.int8)
    V8 = np.ascontiguousarray(V8, np.int8)
    kvp = np.ascontiguousarray(kvp, np.int32)
    ctx, d = K8.shape
    o = np.empty(d, np.int32)
    P = np.empty(ctx, np.int32)
    sig = C.c_int64(0)
    lib().or_attention_row(_p(q8, C.c_int8), C.c_int32(int(mq)), C.c_int32(int(kq)),
                           _p(K8, C.c_int8), _p(V8, C.c_int8), C.c_int(ctx), C.c_int(d),
                           _p(kvp, C.c_int32), _p(o, C.c_int32), _p(P, C.c_int32), C.byref(sig))
    check()
    return o, P, int(sig.value)


def argmax(x):
    x = np.ascontiguousarray(x, np.int32)
    return int(lib().or_argmax(_p(x, C.c_int32), C.c_int(x.size)))


def splitmix64(seed: int, counter: int) -> int:
    return int(lib().or_splitmix64(C.c_uint64(seed), C.c_uint64(counter)))


def sample(logits, inv_temp: int = 65536, top_k: int = 0, top_p: int = 65536, seed: int = 0,
           counter: int = 0) -> int:
    """Integer sampling of one logits row (temperature Q16 inverse, top-k,
    top-p Q16, SplitMix64 draw); returns the token index."""
    x = np.ascontiguousarray(logits, np.int32)
    tok = lib().or_sample(_p(x, C.c_int32), x.size, int(inv_temp), int(top_k), int(top_p),
                          C.c_uint64(seed), C.c_uint64(counter))
    check()
    return int(tok)


def sample_set(logits, inv_temp: int = 65536, top_k: int = 0, top_p: int = 65536):
    """Kept set (bool [n]), weights E (int64 [n]) and their kept sum S."""
    x = np.ascontiguousarray(logits, np.int32)
    keep = np.zeros(x.size, np.uint8)
    E = np.zeros(x.size, np.int64)
    S = C.c_int64(0)
    lib().or_sample_set(_p(x, C.c_int32), x.size, int(inv_temp), int(top_k), int(top_p),
                        keep.ctypes.data_as(C.POINTER(C.c_char)), _p(E, C.c_int64), C.byref(S))
    check()
    return keep.astype(bool), E, int(S.value)


# --------------------------------------------------------------------- model
class Model:
    """A loaded artifact plus per-sequence int8 KV caches, in plain C."""

    def __init__(self, path: str):
        L = lib()
        err = C.c_int(0)
        self._h = L.or_model_load(path.encode(), C.byref(err))
        if not self._h:
            raise OracleError(f"oracle could not load {path} (code {err.value})")
        info = np.zeros(16, np.int32)
        L.or_model_info(self._h, _p(info, C.c_int32))
        (self.n_layers, self.hidden, self.n_q, self.n_kv, self.head_dim, self.ffn,
         self.vocab, self.max_pos, self.qk_norm, self.wbits) = [int(v) for v in info[:10]]

    def close(self):
        if self._h:
            lib().or_model_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_seq(self, max_ctx: int) -> "Seq":
        return Seq(self, max_ctx)


class Seq:
    def __init__(self, model: Model, max_ctx: int):
        self.model = model
        self._h = lib().or_seq_new(model._h, int(max_ctx))

    def __del__(self):
        try:
            if self._h:
                lib().or_seq_free(self._h)
                self._h = None
        except Exception:
            pass

    def __len__(self):
        return int(lib().or_seq_len(self._h))

    def feed(self, tokens, want_hidden: bool = False):
        """Feed tokens in order; returns (argmax, logits int32[V]) of the last
        one, plus the residual after each layer ([L+1, H]) if asked."""
        t = np.ascontiguousarray(np.atleast_1d(tokens), np.int32)
        logits = np.empty(self.model.vocab, np.int32)
        hid = np.empty((self.model.n_layers + 1, self.model.hidden), np.int32) if want_hidden else None
        am = lib().or_seq_feed(self.model._h, self._h, C.c_int(t.size), _p(t, C.c_int32),
                               _p(logits, C.c_int32),
                               _p(hid, C.c_int32) if hid is not None else None)
        check()
        if want_hidden:
            return int(am), logits, hid
        return int(am), logits


def chain_hash(rows, prev: bytes | None = None) -> bytes:
    """SHA-256 chain over int32 rows (little-endian), starting from 32 zero bytes."""
    import hashlib
    h = prev if prev is not None else b"\0" * 32
    for r in rows:
        h = hashlib.sha256(h + np.ascontiguousarray(r, dtype="<i4").tobytes()).digest()
    return h
