"""A float64 restatement of the real-valued decoder that the integer method
approximates (RMSNorm, QK-norm, RoPE, softmax attention with GQA, SwiGLU,
tied lm_head), run on the dequantised artifact weights.

It shares nothing with the oracle: it parses the artifact with numpy from the
format description and uses float64 math throughout. Tests compare the
oracle's integer logits with it to pin the composition of the integer ops
(operand orientation, head mapping, RoPE pairing and sign, residual wiring).
"""
import math
import struct

import numpy as np


def load(path):
    with open(path, "rb") as f:
        blob = f.read()
    assert blob[:8] == b"DETINT01"
    (ver, L, H, nq, nkv, d, F, V, max_pos, qk_norm, eps_h, eps_qk) = struct.unpack("<12i", blob[8:56])
    seed, theta = struct.unpack("<qq", blob[56:72])
    # version 2: 16-bit weights (the exact mode's wide weights), scale m / 2^30
    wide = ver == 2 and struct.unpack("<i", blob[72:76])[0] == 16
    wt, kc = (np.int16, 30) if wide else (np.int8, 22)
    cur = [256]

    def take(dtype, shape):
        cur[0] = (cur[0] + 255) // 256 * 256
        n = int(np.prod(shape))
        a = np.frombuffer(blob, dtype=dtype, count=n, offset=cur[0]).reshape(shape)
        cur[0] += n * np.dtype(dtype).itemsize
        return a

    art = dict(L=L, H=H, nq=nq, nkv=nkv, d=d, F=F, V=V, max_pos=max_pos, qk_norm=qk_norm,
               eps=eps_h / 2.0 ** 32, theta=theta, kc=kc)
    art["embed"] = take(wt, (V, H))
    art["embed_m"] = take(np.int32, (V,))
    art["final_gamma"] = take(np.int16, (H,))
    art["rope_cos"] = take(np.int16, (max_pos, d // 2))
    art["rope_sin"] = take(np.int16, (max_pos, d // 2))
    layers = []
    nqkv = (nq + 2 * nkv) * d
    for _ in range(L):
        ly = {}
        ly["attn_gamma"] = take(np.int16, (H,))
        ly["ffn_gamma"] = take(np.int16, (H,))
        ly["q_gamma"] = take(np.int16, (d,))
        ly["k_gamma"] = take(np.int16, (d,))
        ly["w_qkv"] = take(wt, (nqkv, H))
        ly["m_qkv"] = take(np.int32, (nqkv,))
        ly["w_o"] = take(wt, (H, nq * d))
        ly["m_o"] = take(np.int32, (H,))
        ly["w_gate"] = take(wt, (F, H))
        ly["m_gate"] = take(np.int32, (F,))
        ly["w_up"] = take(wt, (F, H))
        ly["m_up"] = take(np.int32, (F,))
        ly["w_down"] = take(wt, (H, F))
        ly["m_down"] = take(np.int32, (H,))
        ly["kvp"] = take(np.int32, (nkv, 8 + d // 2))
        layers.append(ly)
    art["layers"] = layers
    return art


def _w(w, m, kc=22):
    return w.astype(np.float64) * (m.astype(np.float64) / 2.0 ** kc)[:, None]


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def forward(art, tokens):
    """float64 logits [T, V] for one sequence of token ids (positions 0..T-1)."""
    L, H, nq, nkv, d = art["L"], art["H"], art["nq"], art["nkv"], art["d"]
    eps = art["eps"]
    T = len(tokens)
    grp = nq // nkv
    kc = art["kc"]
    E = _w(art["embed"], art["embed_m"], kc)
    h = E[np.asarray(tokens)]
    half = d // 2
    inv = float(art["theta"]) ** (-2.0 * np.arange(half) / d)
    ang = np.arange(T)[:, None] * inv[None, :]
    cos, sin = np.cos(ang), np.sin(ang)

    def rope(x):  # x [T, heads, d]
        a, b = x[..., :half], x[..., half:]
        c, s = cos[:, None, :], sin[:, None, :]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)

    for ly in art["layers"]:
        y = _rms(h, ly["attn_gamma"] / 4096.0, eps)
        qkv = y @ _w(ly["w_qkv"], ly["m_qkv"], kc).T
        q = qkv[:, : nq * d].reshape(T, nq, d)
        k = qkv[:, nq * d: (nq + nkv) * d].reshape(T, nkv, d)
        v = qkv[:, (nq + nkv) * d:].reshape(T, nkv, d)
        if art["qk_norm"]:
            q = _rms(q, ly["q_gamma"] / 4096.0, eps)
            k = _rms(k, ly["k_gamma"] / 4096.0, eps)
        q, k = rope(q), rope(k)
        o = np.zeros((T, nq, d))
        mask = np.tril(np.ones((T, T), bool))
        for hq in range(nq):
            g = hq // grp
            s = q[:, hq, :] @ k[:, g, :].T / math.sqrt(d)
            s = np.where(mask, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            o[:, hq, :] = p @ v[:, g, :]
        h = h + o.reshape(T, nq * d) @ _w(ly["w_o"], ly["m_o"], kc).T
        y = _rms(h, ly["ffn_gamma"] / 4096.0, eps)
        gt = y @ _w(ly["w_gate"], ly["m_gate"], kc).T
        up = y @ _w(ly["w_up"], ly["m_up"], kc).T
        s = gt / (1.0 + np.exp(-gt)) * up
        h = h + s @ _w(ly["w_down"], ly["m_down"], kc).T
    y = _rms(h, art["final_gamma"] / 4096.0, eps)
    return y @ E.T
