"""ctypes binding of libdetint (include/detint.h), with the same names.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels behind the C ABI. PyTorch supplies device memory and streams. If the
library is missing or cannot be loaded, every entry point raises; there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import hashlib
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdetint.so")
_lib = None

ERRORS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "token id outside the vocabulary",
          4: "context capacity exceeded", 5: "unreadable or malformed artifact",
          6: "artifact sha256 mismatch", 7: "CUDA error", 8: "device out of memory",
          9: "bad sequence id", 10: "saturation recorded"}

# every entry point of include/detint.h
SYMBOLS = ["detint_load", "detint_prefill", "detint_decode_step", "detint_gemm_i8",
           "detint_reset_seq", "detint_seq_len", "detint_status", "detint_set_graph",
           "detint_set_option", "detint_argmax_noalloc", "detint_sample", "detint_fork_seq", "detint_gemm_w16", "detint_split_w16",
           "detint_int8_peak_loop", "detint_model_info", "detint_free", "detint_strerror", "detint_last_error"]


class DetintError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({detail})" if detail else
                         f"{where}: {ERRORS.get(code, code)}")


def lib():
    """The loaded libdetint; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "deterministic_integer_only_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        vp, i32p = C.c_void_p, C.POINTER(C.c_int32)
        L.detint_load.argtypes = [C.c_char_p, C.c_int, C.c_int, vp, C.POINTER(vp)]
        L.detint_prefill.argtypes = [vp, C.c_int, i32p, i32p, vp, vp, vp, vp]
        L.detint_decode_step.argtypes = [vp, C.c_int, i32p, vp, vp, vp, vp]
        L.detint_gemm_i8.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, vp]
        L.detint_reset_seq.argtypes = [vp, C.c_int]
        L.detint_seq_len.argtypes = [vp, C.c_int, i32p]
        L.detint_status.argtypes = [vp, i32p, vp]
        L.detint_set_graph.argtypes = [vp, C.c_int]
        L.detint_set_option.argtypes = [vp, C.c_int, C.c_int]
        L.detint_argmax_noalloc.argtypes = [vp, C.c_int, C.c_int, vp, vp]
        L.detint_fork_seq.argtypes = [vp, C.c_int, C.c_int, C.c_int, vp]
        L.detint_gemm_w16.argtypes = [vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, vp]
        L.detint_split_w16.argtypes = [vp, vp, vp, C.c_longlong, vp]
        L.detint_sample.argtypes = [vp, C.c_int, C.c_int, C.POINTER(SamplingParams), vp, vp]
        L.detint_int8_peak_loop.argtypes = [C.c_int, C.c_int, C.c_int, vp, C.POINTER(C.c_longlong), vp]
        L.detint_model_info.argtypes = [vp, i32p]
        L.detint_free.argtypes = [vp]
        L.detint_free.restype = None
        L.detint_strerror.restype = C.c_char_p
        L.detint_strerror.argtypes = [C.c_int]
        L.detint_last_error.restype = C.c_char_p
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise DetintError(rc, where, lib().detint_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def detint_gemm_i8(A, B, C_out, stream=None):
    """C_out[M,N] (int32, cuda) = A[M,K] (int8) @ B[N,K]^T (int8), exact."""
    M, K = A.shape
    N = B.shape[0]
    _check(lib().detint_gemm_i8(_ptr(A), _ptr(B), _ptr(C_out), M, N, K, _stream(stream)),
           "detint_gemm_i8")
    return C_out


def detint_argmax_noalloc(logits, out, stream=None):
    """out[r] = tie-low argmax of logits[r] (int32 cuda tensors), computed
    without any device allocation (partials in a fixed device array)."""
    import torch
    rows, n = logits.shape
    if logits.dtype != torch.int32 or out.dtype != torch.int32 or not logits.is_cuda or not out.is_cuda:
        raise ValueError("detint_argmax_noalloc: int32 cuda tensors expected")
    if not logits.is_contiguous() or not out.is_contiguous() or out.numel() < rows:
        raise ValueError("detint_argmax_noalloc: contiguous logits [rows, n] and out [rows] expected")
    _check(lib().detint_argmax_noalloc(_ptr(logits), rows, n, _ptr(out), _stream(stream)),
           "detint_argmax_noalloc")
    return out


class SamplingParams(C.Structure):
    """detint_sampling_t: seed, counter (SplitMix64 draw index), inv_temp
    (Q16 of 1/T), top_k (0: off), top_p (Q16, 65536: off)."""
    _fields_ = [("seed", C.c_uint64), ("counter", C.c_uint64), ("inv_temp", C.c_int32),
                ("top_k", C.c_int32), ("top_p", C.c_int32), ("reserved", C.c_int32)]


def detint_sample(logits, params, out=None, stream=None):
    """One integer-sampled token per row of an int32 cuda tensor [rows, n];
    params: one dict (or SamplingParams) per row, or one for every row."""
    import torch
    rows, n = logits.shape
    if isinstance(params, (dict, SamplingParams)):
        params = [params] * rows
    arr = (SamplingParams * rows)()
    for r, p in enumerate(params):
        if isinstance(p, SamplingParams):
            arr[r] = p
        else:
            arr[r] = SamplingParams(int(p.get("seed", 0)), int(p.get("counter", 0)),
                                    int(p.get("inv_temp", 65536)), int(p.get("top_k", 0)),
                                    int(p.get("top_p", 65536)), 0)
    if out is None:
        out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    _check(lib().detint_sample(_ptr(logits), rows, n, arr, _ptr(out), _stream(stream)), "detint_sample")
    return out


def detint_split_w16(W, stream=None):
    """(w_hi int8, w_lo uint8) limbs of an int16 cuda tensor, W = 256 hi + lo."""
    import torch
    hi = torch.empty(W.shape, dtype=torch.int8, device=W.device)
    lo = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    _check(lib().detint_split_w16(_ptr(W), _ptr(hi), _ptr(lo), W.numel(), _stream(stream)), "detint_split_w16")
    return hi, lo


def detint_gemm_w16(A, w_hi, w_lo, C=None, stream=None):
    """C = A @ W.T exactly in int64 (int8 A [M, K], W = 256 w_hi + w_lo [N, K])."""
    import torch
    M, K = A.shape
    N = w_hi.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.int64, device=A.device)
    _check(lib().detint_gemm_w16(_ptr(A), _ptr(w_hi), _ptr(w_lo), _ptr(C), M, N, K, _stream(stream)),
           "detint_gemm_w16")
    return C


def detint_int8_peak_loop(kind: int, blocks: int, iters: int, sink, stream=None) -> int:
    """Launch the integer-pipe peak loop (kind 0 mma.sync s8, 1 dp4a); returns
    the integer operations it performs."""
    ops = C.c_longlong(0)
    _check(lib().detint_int8_peak_loop(int(kind), int(blocks), int(iters), _ptr(sink), C.byref(ops),
                                       _stream(stream)), "detint_int8_peak_loop")
    return int(ops.value)


def chain_hash(rows, prev: bytes | None = None) -> bytes:
    """SHA-256 chain over int32 rows (little-endian) from 32 zero bytes
    (DetLLM README, "Demo": the per-step logits chain hash)."""
    h = prev if prev is not None else b"\0" * 32
    for r in rows:
        h = hashlib.sha256(h + np.ascontiguousarray(r, dtype="<i4").tobytes()).digest()
    return h


class Model:
    """A loaded integer model on the current CUDA device (detint_load)."""

    def __init__(self, path: str, max_batch: int, max_ctx: int, stream=None):
        import torch
        self.torch = torch
        self.stream = stream if stream is not None else torch.cuda.Stream()
        h = C.c_void_p()
        _check(lib().detint_load(path.encode(), int(max_batch), int(max_ctx),
                                 self.stream.cuda_stream, C.byref(h)), "detint_load")
        self._h = h
        info = np.zeros(16, np.int32)
        _check(lib().detint_model_info(self._h, info.ctypes.data_as(C.POINTER(C.c_int32))),
               "detint_model_info")
        (self.n_layers, self.hidden, self.n_q, self.n_kv, self.head_dim, self.ffn, self.vocab,
         self.max_pos, self.qk_norm, self.max_batch, self.max_ctx) = [int(v) for v in info[:11]]

    def close(self):
        if getattr(self, "_h", None):
            lib().detint_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_graph(self, enable: bool):
        _check(lib().detint_set_graph(self._h, int(bool(enable))), "detint_set_graph")

    def set_fused_decode(self, enable: bool):
        _check(lib().detint_set_option(self._h, 1, int(bool(enable))), "detint_set_option")

    def set_staged_decode(self, enable: bool):
        _check(lib().detint_set_option(self._h, 3, int(bool(enable))), "detint_set_option")

    def set_persistent(self, enable: bool):
        _check(lib().detint_set_option(self._h, 4, int(bool(enable))), "detint_set_option")

    def set_wait_test(self, polls: int):
        """While polls > 0, the one-launch decode step's final wait expects a
        tag no CTA writes and gives up after `polls` polls (status slot 6)."""
        _check(lib().detint_set_option(self._h, 5, int(polls)), "detint_set_option")

    def set_tc_prefill(self, enable: bool):
        _check(lib().detint_set_option(self._h, 2, int(bool(enable))), "detint_set_option")

    def reset_seq(self, seq_id: int):
        _check(lib().detint_reset_seq(self._h, int(seq_id)), "detint_reset_seq")

    def fork_seq(self, src: int, dst: int, n_tokens: int):
        """dst starts with src's first n_tokens positions (shared KV blocks)."""
        _check(lib().detint_fork_seq(self._h, int(src), int(dst), int(n_tokens), self.stream.cuda_stream),
               "detint_fork_seq")

    def seq_len(self, seq_id: int) -> int:
        v = C.c_int32()
        _check(lib().detint_seq_len(self._h, int(seq_id), C.byref(v)), "detint_seq_len")
        return int(v.value)

    def status(self) -> np.ndarray:
        flags = np.zeros(8, np.int32)
        lib().detint_status(self._h, flags.ctypes.data_as(C.POINTER(C.c_int32)),
                            self.stream.cuda_stream)
        return flags

    def prefill(self, seq_ids, tokens, cu_lens, logits=None, next_tok=None):
        """tokens: int32 cuda tensor (ragged, concatenated); cu_lens: host ints."""
        torch = self.torch
        seq = _i32(seq_ids)
        cu = _i32(cu_lens)
        n = seq.size
        if next_tok is None:
            next_tok = torch.empty(n, dtype=torch.int32, device=tokens.device)
        _check(lib().detint_prefill(self._h, n, seq.ctypes.data_as(C.POINTER(C.c_int32)),
                                    cu.ctypes.data_as(C.POINTER(C.c_int32)), _ptr(tokens),
                                    _ptr(logits), _ptr(next_tok), self.stream.cuda_stream),
               "detint_prefill")
        return next_tok

    def decode_step(self, seq_ids, tok, logits=None, next_tok=None):
        torch = self.torch
        seq = _i32(seq_ids)
        if next_tok is None:
            next_tok = torch.empty(seq.size, dtype=torch.int32, device=tok.device)
        _check(lib().detint_decode_step(self._h, seq.size, seq.ctypes.data_as(C.POINTER(C.c_int32)),
                                        _ptr(tok), _ptr(logits), _ptr(next_tok),
                                        self.stream.cuda_stream), "detint_decode_step")
        return next_tok

    def generate(self, prompts, max_new: int, seq_ids=None, keep_logits: bool = True, sampling=None):
        """Decode a ragged batch of prompts (lists of ids), greedy by default.

        Returns (tokens [B][max_new] int32 numpy, logits rows per step (list of
        [B, V] numpy arrays) or chain-hash digests per row when keep_logits is
        "hash"). Step 0 is the prefill's last-position logits (README, "Usage":
        generate(ids, max_new)). sampling: None (greedy) or a dict of
        detint_sample parameters (seed, inv_temp, top_k, top_p) or one dict per
        row; step s of row b draws with counter = s, so a row's tokens do not
        depend on the rest of the batch.
        """
        torch = self.torch
        B = len(prompts)
        seq_ids = list(range(B)) if seq_ids is None else list(seq_ids)
        dev = torch.device("cuda")
        cu = np.zeros(B + 1, np.int64)
        cu[1:] = np.cumsum([len(p) for p in prompts])
        flat = torch.tensor(np.concatenate([np.asarray(p, np.int32) for p in prompts]),
                            dtype=torch.int32, device=dev)
        logits = torch.empty((B, self.vocab), dtype=torch.int32, device=dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        toks = np.zeros((B, max_new), np.int32)
        rows = []
        hashes = [b"\0" * 32] * B
        if sampling is not None:
            per_row = sampling if isinstance(sampling, (list, tuple)) else [sampling] * B
        with torch.cuda.stream(self.stream):
            self.prefill(seq_ids, flat, cu, logits, tok)
            for step in range(max_new):
                if step:
                    self.decode_step(seq_ids, tok, logits, tok)
                if sampling is not None:
                    detint_sample(logits, [dict(p, counter=step) for p in per_row], out=tok,
                                  stream=self.stream)
                lg = logits.cpu().numpy()
                toks[:, step] = tok.cpu().numpy()
                if keep_logits == "hash":
                    hashes = [chain_hash([lg[b]], hashes[b]) for b in range(B)]
                elif keep_logits:
                    rows.append(lg)
        self.stream.synchronize()
        return toks, (hashes if keep_logits == "hash" else rows)
