"""detint for GB300: the integer-only LLM decoder forward pass on sm_103a.

The compute path is libdetint (hand-written CUDA kernels behind the C ABI in
include/detint.h); this package only marshals arguments to it.
"""
from .binding import (Model, DetintError, chain_hash, detint_gemm_i8, detint_argmax_noalloc,
                      detint_sample, SamplingParams, detint_gemm_w16, detint_split_w16, detint_int8_peak_loop, lib,
                      LIB_PATH, SYMBOLS)

__all__ = ["Model", "DetintError", "chain_hash", "detint_gemm_i8", "detint_argmax_noalloc",
           "detint_sample", "SamplingParams", "detint_gemm_w16", "detint_split_w16", "detint_int8_peak_loop", "lib",
           "LIB_PATH", "SYMBOLS"]
