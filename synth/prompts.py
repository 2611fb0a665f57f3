"""Seeded prompt ids and co-prompt lengths.

The DetLLM demo prompt (the first 64 tokens of a sonnet) and its junk
co-prompts are replaced by token ids drawn uniformly from the vocabulary with
a stated seed; there is no tokenizer or text here.
"""
import numpy as np

_PROMPT_TAG = 0x70726F6D  # "prom"
_COLEN_TAG = 0x636F6C6E   # "coln"


def prompt_ids(seed: int, index: int, length: int, vocab: int) -> np.ndarray:
    """Token ids of prompt `index` for `seed`: int32[length], uniform in [0, vocab)."""
    rng = np.random.default_rng([seed, _PROMPT_TAG, index])
    return rng.integers(0, vocab, size=length, dtype=np.int64).astype(np.int32)


def coprompt_lengths(seed: int, n: int, lo: int = 16, hi: int = 256) -> np.ndarray:
    """Lengths of `n` co-prompts, uniform in [lo, hi] (inclusive)."""
    rng = np.random.default_rng([seed, _COLEN_TAG])
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)
