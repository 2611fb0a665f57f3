"""Seeded synthetic int8 model artifacts (format: the artifact section of the
arithmetic specification in docs/), and their wide-weight (int16) variants
for the exact mode.

Three shapes: a tiny Qwen3-style model, a Qwen3-0.6B-shaped model and a
Llama-3.2-1B-shaped model. One numpy PCG64 stream per artifact draws every
random section in file order. The K/V scales and the per-channel key shifts
are the offline calibration stand-in: they are derived in float64 from the
drawn weights and gammas (expected channel RMS of a unit-RMS input, clipped at
four standard deviations), never from running the model.

A wide artifact (version 2, 16-bit weights) of the same shape and seed holds
w16 = 256 w8 + r for every linear and embedding weight, with w8 the int8
artifact's weight and r uniform in [-127, 127] from a second PCG64 stream
(seed + WIDE_SEED_OFFSET) drawn in file order; every other section is the
int8 artifact's. Rounding w16 / 256 to the nearest integer gives back w8, so
the int8 artifact is the int8 rounding of the wide one.
"""
from __future__ import annotations

import hashlib
import math
import os
import struct
from dataclasses import dataclass

import numpy as np

MAGIC = b"DETINT01"
VERSION = 1
VERSION_WIDE = 2
WIDE_SEED_OFFSET = 0x5EED0016
ALIGN = 256
HEADER_BYTES = 256
CLIP_SIGMAS = 4.0


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    max_pos: int
    qk_norm: int
    rope_theta: int
    eps: float

    @property
    def n_qkv(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim


MODEL_SHAPES = {
    # 2 layers, hidden 256, 4 q / 2 kv heads, head_dim 64, FFN 768, vocab 1024.
    "tiny": ModelShape("tiny", 2, 256, 4, 2, 64, 768, 1024, 1024, 1, 1_000_000, 1e-6),
    # Qwen3-0.6B shape: 28 layers, hidden 1024, 16 q / 8 kv, head_dim 128,
    # FFN 3072, vocab 151936, QK-norm, theta 1e6.
    "qwen3-0.6b": ModelShape("qwen3-0.6b", 28, 1024, 16, 8, 128, 3072, 151936,
                             8192, 1, 1_000_000, 1e-6),
    # Llama-3.2-1B shape: 16 layers, hidden 2048, 32 q / 8 kv, head_dim 64,
    # FFN 8192, vocab 128256, no QK-norm, theta 5e5 (the pages do not state it).
    "llama-1b": ModelShape("llama-1b", 16, 2048, 32, 8, 64, 8192, 128256,
                           4096, 0, 500_000, 1e-5),
}


def _pad(f, written: int) -> int:
    rem = (-written) % ALIGN
    if rem:
        f.write(b"\0" * rem)
    return written + rem


def _dyadic_real(x: float) -> tuple[int, int]:
    """(m, k) with m/2^k ~= x and m in [2^14, 2^15] (offline, float64)."""
    assert x > 0.0
    k = 14 - math.floor(math.log2(x))
    m = int(round(x * 2.0 ** k))
    if m < 2 ** 14:
        k += 1
        m = int(round(x * 2.0 ** k))
    if m > 2 ** 15:
        k -= 1
        m = int(round(x * 2.0 ** k))
    assert 2 ** 14 <= m <= 2 ** 15, (x, m, k)
    return m, k


class _Writer:
    def __init__(self, f):
        self.f = f
        self.pos = 0
        self.h = hashlib.sha256()

    def write(self, b: bytes):
        self.f.write(b)
        self.h.update(b)
        self.pos += len(b)

    def section(self, arr: np.ndarray):
        rem = (-self.pos) % ALIGN
        if rem:
            self.write(b"\0" * rem)
        self.write(np.ascontiguousarray(arr).tobytes())


def _int8_weights(rng, rows: int, cols: int, chunk_rows: int | None = None) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.int8)
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 24) // cols)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        z = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        z *= np.float32(24.0)
        np.rint(z, out=z)
        np.clip(z, -127, 127, out=z)
        out[r0:r1] = z.astype(np.int8)
    return out


def _scales(rng, n: int) -> np.ndarray:
    return rng.integers(1 << 14, 1 << 15, size=n, dtype=np.int64).astype(np.int32)


def _gammas(rng, n: int) -> np.ndarray:
    return rng.integers(1 << 11, 1 << 13, size=n, dtype=np.int64).astype(np.int16)


def rope_tables(shape: ModelShape) -> tuple[np.ndarray, np.ndarray]:
    """int16 Q14 cos/sin tables [max_pos, d/2], built once in float64."""
    half = shape.head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = float(shape.rope_theta) ** (-2.0 * i / shape.head_dim)
    p = np.arange(shape.max_pos, dtype=np.float64)[:, None]
    ang = p * inv_freq[None, :]
    c = np.rint(np.cos(ang) * 16384.0).astype(np.int16)
    s = np.rint(np.sin(ang) * 16384.0).astype(np.int16)
    return c, s


def _kv_params(shape: ModelShape, attn_gamma, k_gamma, w_qkv, m_qkv) -> np.ndarray:
    d, half, nq, nkv = shape.head_dim, shape.head_dim // 2, shape.n_q, shape.n_kv
    rms_y = math.sqrt(float(np.mean((attn_gamma.astype(np.float64) / 4096.0) ** 2)))
    out = np.zeros((nkv, 8 + half), dtype=np.int32)
    for g in range(nkv):
        rk = slice((nq + g) * d, (nq + g + 1) * d)
        rv = slice((nq + nkv + g) * d, (nq + nkv + g + 1) * d)
        wk = w_qkv[rk].astype(np.float64)
        wv = w_qkv[rv].astype(np.float64)
        sk = rms_y * np.sqrt((wk * wk).sum(1)) * m_qkv[rk].astype(np.float64) / 2.0 ** 22
        sv = rms_y * np.sqrt((wv * wv).sum(1)) * m_qkv[rv].astype(np.float64) / 2.0 ** 22
        if shape.qk_norm:
            sk = (k_gamma.astype(np.float64) / 4096.0) * sk / math.sqrt(float(np.mean(sk * sk)))
        rho = np.sqrt((sk[:half] ** 2 + sk[half:] ** 2) / 2.0)
        e = np.minimum(3, np.floor(np.log2(rho.max() / rho))).astype(np.int64)
        e = np.maximum(e, 0)
        big_e = int(e.max())
        s_k = CLIP_SIGMAS * float((rho * 2.0 ** e).max()) / 127.0
        s_v = CLIP_SIGMAS * float(sv.max()) / 127.0
        kqm, kqs = _dyadic_real(1.0 / (s_k * 2.0 ** 14))
        vqm, vqs = _dyadic_real(1.0 / (s_v * 2.0 ** 12))
        mv, kv = _dyadic_real(s_v)
        cstm, cstk = _dyadic_real(s_k * 2.0 ** (-big_e) * math.log2(math.e) / math.sqrt(d))
        out[g, :8] = [kqm, kqs, vqm, vqs, mv, kv, cstm, cstk]
        out[g, 8:] = e
    return out


def header_bytes(shape: ModelShape, seed: int, wide: bool = False) -> bytes:
    eps_h = int(round(shape.eps * 2.0 ** 32))
    eps_qk = int(round(shape.eps * 2.0 ** 24))
    hdr = MAGIC + struct.pack("<12i", VERSION_WIDE if wide else VERSION, shape.n_layers, shape.hidden,
                              shape.n_q, shape.n_kv, shape.head_dim, shape.ffn, shape.vocab,
                              shape.max_pos, shape.qk_norm, eps_h, eps_qk)
    hdr += struct.pack("<qq", seed, shape.rope_theta)
    assert len(hdr) == 72
    if wide:
        hdr += struct.pack("<i", 16)                 # weight bits
    return hdr + b"\0" * (HEADER_BYTES - len(hdr))


def _widen(rng2, w8: np.ndarray, chunk: int = 1 << 24) -> np.ndarray:
    """w16 = 256 w8 + r, r uniform in [-127, 127] (row chunks, file order)."""
    out = np.empty(w8.shape, dtype=np.int16)
    flat_in, flat_out = w8.reshape(-1), out.reshape(-1)
    for i0 in range(0, flat_in.size, chunk):
        i1 = min(flat_in.size, i0 + chunk)
        r = rng2.integers(-127, 128, size=i1 - i0, dtype=np.int64)
        flat_out[i0:i1] = (flat_in[i0:i1].astype(np.int64) * 256 + r).astype(np.int16)
    return out


def write_artifact(path: str, shape: ModelShape | str, seed: int, wide: bool = False) -> str:
    """Write the artifact for `shape` and `seed` to `path` plus `path.sha256`
    (the wide variant with 16-bit weights when `wide`).

    Returns the hex SHA-256 of the file.
    """
    if isinstance(shape, str):
        shape = MODEL_SHAPES[shape]
    rng = np.random.Generator(np.random.PCG64(seed))
    rng2 = np.random.Generator(np.random.PCG64(seed + WIDE_SEED_OFFSET)) if wide else None

    def wsec(w8):
        return _widen(rng2, w8) if wide else w8

    H, F, V, d = shape.hidden, shape.ffn, shape.vocab, shape.head_dim
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        w = _Writer(f)
        w.write(header_bytes(shape, seed, wide))
        w.section(wsec(_int8_weights(rng, V, H)))    # embed
        w.section(_scales(rng, V))                   # embed_m
        w.section(_gammas(rng, H))                   # final_gamma
        cos, sin = rope_tables(shape)
        w.section(cos)
        w.section(sin)
        for _ in range(shape.n_layers):
            attn_gamma = _gammas(rng, H)
            ffn_gamma = _gammas(rng, H)
            q_gamma = _gammas(rng, d)
            k_gamma = _gammas(rng, d)
            w_qkv = _int8_weights(rng, shape.n_qkv, H)
            m_qkv = _scales(rng, shape.n_qkv)
            w_o = _int8_weights(rng, H, shape.n_q * d)
            m_o = _scales(rng, H)
            w_gate = _int8_weights(rng, F, H)
            m_gate = _scales(rng, F)
            w_up = _int8_weights(rng, F, H)
            m_up = _scales(rng, F)
            w_down = _int8_weights(rng, H, F)
            m_down = _scales(rng, H)
            kvp = _kv_params(shape, attn_gamma, k_gamma, w_qkv, m_qkv)
            for arr in (attn_gamma, ffn_gamma, q_gamma, k_gamma, wsec(w_qkv), m_qkv, wsec(w_o), m_o,
                        wsec(w_gate), m_gate, wsec(w_up), m_up, wsec(w_down), m_down, kvp):
                w.section(arr)
        rem = (-w.pos) % ALIGN
        if rem:
            w.write(b"\0" * rem)
        digest = w.h.hexdigest()
    os.replace(tmp, path)
    with open(path + ".sha256", "w") as f:
        f.write(digest + "\n")
    return digest


def read_header(path: str) -> dict:
    with open(path, "rb") as f:
        b = f.read(HEADER_BYTES)
    if b[:8] != MAGIC:
        raise ValueError("not a detint artifact")
    v = struct.unpack("<12i", b[8:56])
    seed, theta = struct.unpack("<qq", b[56:72])
    wbits = struct.unpack("<i", b[72:76])[0] if v[0] == VERSION_WIDE else 8
    keys = ["version", "n_layers", "hidden", "n_q", "n_kv", "head_dim", "ffn", "vocab",
            "max_pos", "qk_norm", "eps_h", "eps_qk"]
    d = dict(zip(keys, v))
    d["seed"] = seed
    d["rope_theta"] = theta
    d["wbits"] = wbits
    return d


def artifact_path(shape: str, seed: int, root: str | None = None, wide: bool = False) -> str:
    root = root or os.environ.get("DETINT_ARTIFACT_DIR") or os.path.join(
        os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_artifacts")
    os.makedirs(root, exist_ok=True)
    return os.path.join(root, f"{shape}-seed{seed}{'-w16' if wide else ''}.detint")


def ensure_artifact(shape: str, seed: int, root: str | None = None, wide: bool = False) -> str:
    """Path of the artifact for (shape, seed), writing it first if absent
    (the wide variant when `wide`)."""
    p = artifact_path(shape, seed, root, wide)
    if not (os.path.exists(p) and os.path.exists(p + ".sha256")):
        write_artifact(p, shape, seed, wide)
    return p
