"""Plain CPU restatement of the SVDq keys-only low-rank cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): used by the tests,
never by the product path; it shares no code with the CUDA path.

Method source: page "veloxquant_mlx.cache.svdq_cache module", section
"Design" (prefill steps 1-6, decode steps 1-3, "Byte accounting", the
effective key bit-width), and the SVDqKVCache config fields: svdq_rank
(explicit, else energy threshold), svdq_energy_threshold 0.95,
svdq_bit_schedule (8, 4, 2, 1, 1, 0, 0, 0) most significant group first,
svdq_group_size 32 along the token axis.  Values are not compressed.

Readings where the page is silent (also listed in the design notes):
  * Per-head fit.  Each KV head has its own basis and mean, fitted on that
    head's rows over the whole prefill batch (the stacking reading of the
    latent cache with one head per group).  With the energy threshold each
    head keeps its own rank ("each head can land at its own rank").
  * Channel groups.  "Equal-size contiguous groups" when r is not a multiple
    of the schedule's length: group sizes differ by at most one, the larger
    groups first (the most significant channels get the extra channel).
  * Quantizer.  b bits (1..8): the asymmetric min/max quantizer over groups
    of 32 consecutive tokens, with the latent cache's rounding readings (fp16
    scale and zero, codes in fp32 against them, round half to even, a zero
    scale gives code 0).  0 bits: nothing is stored and the channel reads
    back as exactly zero ("0 bits truncates a group to exactly zero").
  * Partial blocks.  As in the latent cache, a 32-token block is quantized
    when its last token arrives; until then its latents wait in fp32.
  * Attention.  Keys are reconstructed as K_hat = L_hat V^T + mean in fp64
    (the page hands fp16 keys to the attention: `fp16_keys=True` rounds
    K_hat to fp16 first); values are used as given (fp16).
"""
from __future__ import annotations

import numpy as np

from .palu_oracle import BLOCK, ENERGY_SIGMA, fit, project

SCHEDULE = (8, 4, 2, 1, 1, 0, 0, 0)
ENERGY_THRESHOLD = 0.95


def channel_bits(r: int, schedule=SCHEDULE) -> np.ndarray:
    """Bit width of each of the r latent channels (most significant first)."""
    n = len(schedule)
    sizes = [r // n + (1 if g < r % n else 0) for g in range(n)]
    return np.repeat(np.asarray(schedule, dtype=np.int64), sizes)


def effective_bits(r: int, D: int, schedule=SCHEDULE) -> float:
    """Code bits per element of the [S, D] key tensor: the sum of the channels'
    widths over D.  Equals the page's (r/D) * mean(schedule) when the
    schedule's length divides r."""
    return float(channel_bits(r, schedule).sum()) / D


def quantize_blocks(L: np.ndarray, bits: np.ndarray):
    """Per-channel widths: L [N, 32, r] fp32 -> codes uint8 [N, 32, r],
    scale fp16 [N, r], zero fp16 [N, r].  A 0-bit channel stores nothing:
    code, scale and zero 0."""
    L = np.asarray(L, dtype=np.float32)
    N, T, r = L.shape
    assert T == BLOCK and len(bits) == r
    bits = np.asarray(bits)
    qmax = (2.0 ** bits - 1).astype(np.float32)              # [r]
    mn = L.min(axis=1)
    mx = L.max(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        scale = ((mx - mn) / qmax).astype(np.float32)         # fp32 subtract, fp32 divide
    kept = bits > 0
    s_h = np.where(kept, scale, 0.0).astype(np.float16)
    z_h = np.where(kept, mn, 0.0).astype(np.float16)
    s32 = s_h.astype(np.float32)[:, None, :]
    z32 = z_h.astype(np.float32)[:, None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((L - z32) / s32)
    q = np.where(s32 == 0, 0.0, q)
    q = np.clip(q, 0.0, qmax[None, None, :])
    return q.astype(np.uint8), s_h, z_h


def dequantize(codes, s_h, z_h) -> np.ndarray:
    """L_hat = code * scale + zero in fp64 ([..., 32, r] codes, [..., r] s/z)."""
    return (codes.astype(np.float64) * s_h.astype(np.float64)[..., None, :]
            + z_h.astype(np.float64)[..., None, :])


def svdq_fit(x: np.ndarray, rank: int = 0, energy_threshold: float = ENERGY_THRESHOLD,
             energy_mode: int = ENERGY_SIGMA):
    """Per-head fit of keys x [B, H, S, D] (prefill steps 1-2).

    Returns (bases, mus, ranks): bases[h] is [D, r_h] fp32 (columns by
    descending singular value, canonical sign), mus [H, D] fp32, ranks [H].
    rank > 0 gives every head that rank; rank == 0 picks each head's own rank
    by the energy threshold.
    """
    H = x.shape[1]
    f = fit(x, n_groups=H, rank=rank, energy_threshold=energy_threshold, energy_mode=energy_mode)
    ranks = [int(r) for r in f.group_ranks]
    bases = [f.basis[h][:, :ranks[h]].astype(np.float32) for h in range(H)]
    return bases, f.mu.astype(np.float32), ranks


class SvdqKeyCache:
    """Key cache of one layer: per head h a basis [D, r_h] and mean [D]; per
    (batch, head) the codes of the full 32-token blocks and the fp32 latents
    of the partial one.  Values are not part of it (kept as fp16)."""

    def __init__(self, bases, mus, B: int, schedule=SCHEDULE):
        self.bases = [np.asarray(b, dtype=np.float32) for b in bases]
        self.mus = np.asarray(mus, dtype=np.float32)
        self.B, self.H = B, len(self.bases)
        self.D = self.mus.shape[1]
        self.schedule = tuple(schedule)
        self.ranks = [b.shape[1] for b in self.bases]
        self.bits = [channel_bits(r, schedule) for r in self.ranks]
        self.codes = [np.zeros((B, 0, BLOCK, r), np.uint8) for r in self.ranks]
        self.scale = [np.zeros((B, 0, r), np.float16) for r in self.ranks]
        self.zero = [np.zeros((B, 0, r), np.float16) for r in self.ranks]
        self.tail = [np.zeros((B, 0, r), np.float32) for r in self.ranks]

    @property
    def length(self) -> int:
        return self.codes[0].shape[1] * BLOCK + self.tail[0].shape[1]

    def append(self, k: np.ndarray) -> None:
        """Append keys k [B, H, T, D] (fp16): project into each head's basis
        (decode step 1), quantize every block that completes."""
        k = np.asarray(k, dtype=np.float16)
        for h in range(self.H):
            L = project(k[:, h], self.bases[h], self.mus[h])          # [B, T, r] fp32
            w = np.concatenate([self.tail[h], L], axis=1)
            n_new = w.shape[1] // BLOCK
            if n_new:
                r = self.ranks[h]
                blocks = w[:, :n_new * BLOCK].reshape(self.B * n_new, BLOCK, r)
                c, s, z = quantize_blocks(blocks, self.bits[h])
                self.codes[h] = np.concatenate([self.codes[h], c.reshape(self.B, n_new, BLOCK, r)], axis=1)
                self.scale[h] = np.concatenate([self.scale[h], s.reshape(self.B, n_new, r)], axis=1)
                self.zero[h] = np.concatenate([self.zero[h], z.reshape(self.B, n_new, r)], axis=1)
            self.tail[h] = w[:, n_new * BLOCK:].copy()

    def latents(self, h: int) -> np.ndarray:
        """Dequantized latents of head h, [B, S, r_h] fp64 (tail exact)."""
        blk = dequantize(self.codes[h], self.scale[h], self.zero[h]).reshape(self.B, -1, self.ranks[h])
        return np.concatenate([blk, self.tail[h].astype(np.float64)], axis=1)

    def keys(self, fp16_keys: bool = False) -> np.ndarray:
        """Reconstructed keys K_hat = L_hat V^T + mean, [B, H, S, D] fp64 (prefill
        step 5); rounded to fp16 with fp16_keys."""
        out = np.stack([self.latents(h) @ self.bases[h].astype(np.float64).T + self.mus[h].astype(np.float64)
                        for h in range(self.H)], axis=1)
        return out.astype(np.float16).astype(np.float64) if fp16_keys else out

    def code_bytes(self) -> float:
        """Bytes of the full blocks' codes at each channel's width (the page's
        latent storage at the schedule's per-group bit rate)."""
        n = self.codes[0].shape[1]
        return float(sum(self.B * n * BLOCK * int(b.sum()) for b in self.bits)) / 8

    def assigned_avg_bits(self) -> float:
        """The page's effective key bit-width, averaged over heads."""
        return float(np.mean([effective_bits(r, self.D, self.schedule) for r in self.ranks]))


# --------------------------------------------------------------------------
# Record layout of a 32-token block of one (batch, head) stream, as stored
# by the GPU cache (a storage format of this build; the page fixes only the
# widths and the LSB-first packing of sub-byte codes).  The kept channels
# (width > 0) come first, each channel's 32 codes packed LSB-first at its
# width (token t at bit t * b of the channel's 4 * b bytes), then one fp16
# (scale, zero) pair per kept channel; the record is padded to 16 bytes.
# --------------------------------------------------------------------------

def record_layout(r: int, schedule=SCHEDULE):
    """(bits [r], kept channels, code byte offset per kept channel,
    byte offset of the scale/zero pairs, record bytes)."""
    bits = channel_bits(r, schedule)
    kept = int((bits > 0).sum())
    ends = np.cumsum(4 * bits[:kept])
    offs = np.concatenate([[0], ends[:-1]]).astype(np.int64) if kept else np.zeros(0, np.int64)
    sz_off = int(ends[-1]) if kept else 0
    return bits, kept, offs, sz_off, -(-(sz_off + 4 * kept) // 16) * 16


def pack_record(codes: np.ndarray, s_h: np.ndarray, z_h: np.ndarray, r: int, stride: int,
                schedule=SCHEDULE) -> np.ndarray:
    """codes [32, r] uint8, scale/zero [r] fp16 -> one record of `stride` bytes."""
    bits, kept, offs, sz_off, nbytes = record_layout(r, schedule)
    assert stride >= nbytes
    rec = np.zeros(stride, np.uint8)
    for j in range(kept):
        b = int(bits[j])
        for t in range(BLOCK):
            pos = t * b
            val = int(codes[t, j]) << (pos % 8)
            for k in range(-(-(pos % 8 + b) // 8)):
                rec[offs[j] + pos // 8 + k] |= (val >> (8 * k)) & 0xFF
    sz = np.stack([np.asarray(s_h, np.float16)[:kept], np.asarray(z_h, np.float16)[:kept]], axis=1)
    rec[sz_off:sz_off + 4 * kept] = sz.view(np.uint8).reshape(-1)
    return rec


def unpack_record(rec: np.ndarray, r: int, schedule=SCHEDULE):
    """One record -> codes [32, r] uint8, scale/zero [r] fp16 (0 for the
    channels that are not stored)."""
    bits, kept, offs, sz_off, _ = record_layout(r, schedule)
    rec = np.asarray(rec, np.uint8)
    codes = np.zeros((BLOCK, r), np.uint8)
    for j in range(kept):
        b = int(bits[j])
        for t in range(BLOCK):
            pos = t * b
            word = 0
            for k in range(-(-(pos % 8 + b) // 8)):
                word |= int(rec[offs[j] + pos // 8 + k]) << (8 * k)
            codes[t, j] = (word >> (pos % 8)) & ((1 << b) - 1)
    sz = rec[sz_off:sz_off + 4 * kept].copy().view(np.float16).reshape(kept, 2)
    s_h = np.zeros(r, np.float16)
    z_h = np.zeros(r, np.float16)
    s_h[:kept], z_h[:kept] = sz[:, 0], sz[:, 1]
    return codes, s_h, z_h


def svdq_attend(q: np.ndarray, kc: SvdqKeyCache, v: np.ndarray, scale: float | None = None,
                fp16_keys: bool = False) -> np.ndarray:
    """Single-token decode attention, fp64: q [B, Hq, D], values v [B, H, S, D]
    (fp16, stored as they came); query head h reads KV head h // (Hq / H)."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Gq = Hq // kc.H
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    K = kc.keys(fp16_keys)
    V = np.asarray(v, dtype=np.float64)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for hq in range(Hq):
            h = hq // Gq
            s = (K[b, h] @ q[b, hq]) * scale
            p = np.exp(s - s.max())
            out[b, hq] = (p @ V[b, h]) / p.sum()
    return out
