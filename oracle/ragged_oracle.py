"""Ragged per-sequence lengths for the latent cache: plain CPU restatement.

TEST INFRASTRUCTURE ONLY (see the package docstring): used by the tests,
never by the product path; it shares no code with the CUDA path.

Why sequences of one batch differ in length (page "add TurboQuant KV cache
compression", the pull request's description and review): prompts of
different lengths share a batch, the prompt cache restores a saved prefix,
speculative decoding rolls back rejected tokens, and multi-turn reuse
continues from earlier state.

Readings (also listed in the design notes):
  * One basis and mean per (layer, tensor, head group), fitted on the prefill
    batch and shared by its sequences, as with uniform lengths.
  * A sequence's KV heads share its length.  Its blocks and its partial-block
    tail follow the uniform cache's rules at its own positions: a block is
    quantized when its own 32nd token arrives.
  * An append gives each sequence its own token count; 0 leaves it unchanged.
  * Decode attention of sequence b covers exactly its own tokens.
  * A per-sequence rollback follows the uniform cache's truncation rule: to a
    block boundary, or inside the current partial block, never reopening a
    quantized block.
"""
from __future__ import annotations

import numpy as np

from .palu_oracle import BLOCK, OracleCache, attend


class RaggedCache:
    """One tensor (K or V) of one layer for B sequences of their own lengths."""

    def __init__(self, role: int, basis, mu, r: int, B: int, Hkv: int, capacity: int, quantize: bool = True):
        self.B, self.Hkv = B, Hkv
        self.seqs = [OracleCache(role, basis, mu, r, 1, Hkv, capacity, quantize) for _ in range(B)]

    @property
    def lengths(self) -> list:
        return [s.length for s in self.seqs]

    def append(self, x: np.ndarray, counts) -> None:
        """x [B, Hkv, T, D] (fp16): sequence b appends its first counts[b] rows."""
        x = np.asarray(x)
        assert x.shape[0] == self.B and len(counts) == self.B
        for b, n in enumerate(counts):
            assert 0 <= n <= x.shape[2]
            if n:
                self.seqs[b].append(x[b:b + 1, :, :n])

    def truncate(self, lengths) -> None:
        """Roll each sequence back to lengths[b] tokens."""
        for s, n in zip(self.seqs, lengths):
            if not 0 <= n <= s.length:
                raise ValueError("a rollback cannot grow a sequence")
            if n % BLOCK and n // BLOCK != s.length // BLOCK:
                raise ValueError("a rollback may not reopen a quantized block")
            s.length = n


def attend_ragged(q: np.ndarray, kc: RaggedCache, vc: RaggedCache, scale: float | None = None) -> np.ndarray:
    """q [B, Hq, D] -> [B, Hq, D] fp64: sequence b attends over its own tokens."""
    q = np.asarray(q)
    assert kc.lengths == vc.lengths
    return np.concatenate([attend(q[b:b + 1], kc.seqs[b], vc.seqs[b], scale) for b in range(kc.B)], axis=0)
