"""Plain CPU restatement of the KIVI-2bit KV cache (the compressed comparator).

TEST INFRASTRUCTURE ONLY (see the package docstring): used by the tests and
the benchmark's CPU-baseline leg, never by the product path; it shares no
code with the CUDA path.

Method source: blog post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What
KIVI is" (and its usage example: bit_width_inlier=2, kivi_group_size=32,
residual_length=32):
  * keys are quantized per channel: one (scale, zero) per (channel, group of
    32 consecutive tokens);
  * values are quantized per token: one (scale, zero) per (token, group of 32
    consecutive channels);
  * the most recent tokens are kept exactly (fp16) in a residual window;
  * the quantizer is the asymmetric min/max group quantizer
        zero = min(g), scale = (max(g) - min(g)) / (2^b - 1),
        q = round((g - zero) / scale),  g_hat = q * scale + zero,
    the same one the latent cache uses (palu_oracle.quantize_blocks, whose
    readings -- fp16 scale and zero, fp32 arithmetic against the stored fp16
    values, round half to even, zero scale gives code 0 -- apply here too).

Reading of the residual window (the page gives only "the last R tokens" and
"quantizes tokens once they age out of that window"): key groups run along
the token axis, so a key group can only be formed from 32 whole tokens.  A
32-token block is therefore quantized -- keys and values together -- when
its 32nd token arrives; the window holds the tokens after the last complete
block (0..31 of them), exactly as they came (fp16).  With R = 32 equal to the
group size this is the window of the page's example that still lets every
key group be complete.

Decode attention is the naive fp64 softmax attention on the dequantized
keys and values (window rows exact), with the GQA mapping query head h ->
KV head h // (Hq / Hkv).
"""
from __future__ import annotations

import numpy as np

from .palu_oracle import BLOCK, quantize_blocks

BITS = 2            # KIVI-2bit: bit_width_inlier = 2
GROUP = 32          # kivi_group_size: tokens per key group, channels per value group


def quantize_keys(K: np.ndarray, bits: int = BITS):
    """Per-channel key quantization of whole blocks.

    K is [N, 32, D] (N blocks of 32 tokens).  Groups run along the token
    axis: one (scale, zero) per (block, channel).
    Returns codes uint8 [N, 32, D], scale fp16 [N, D], zero fp16 [N, D].
    """
    K = np.asarray(K, dtype=np.float32)
    assert K.ndim == 3 and K.shape[1] == BLOCK
    return quantize_blocks(K, n_hi=0, lo_bit=bits)


def quantize_values(V: np.ndarray, bits: int = BITS):
    """Per-token value quantization.

    V is [N, 32, D].  Groups run along the channel axis: one (scale, zero)
    per (token, group of GROUP consecutive channels).
    Returns codes uint8 [N, 32, D], scale fp16 [N, 32, D/GROUP], zero likewise.
    """
    V = np.asarray(V, dtype=np.float32)
    N, T, D = V.shape
    assert D % GROUP == 0
    n_g = D // GROUP
    # every (token, channel group) is one group of GROUP values: lay the groups
    # out as [groups, GROUP, 1] so the quantizer's group axis (axis 1) is the
    # channel axis
    groups = V.reshape(N * T * n_g, GROUP, 1)
    codes, s, z = quantize_blocks(groups, n_hi=0, lo_bit=bits)
    return codes.reshape(N, T, D), s.reshape(N, T, n_g), z.reshape(N, T, n_g)


def dequantize_keys(codes, s, z) -> np.ndarray:
    """[..., 32, D] codes with [..., D] scale/zero -> fp64 keys."""
    return codes.astype(np.float64) * s.astype(np.float64)[..., None, :] + z.astype(np.float64)[..., None, :]


def dequantize_values(codes, s, z) -> np.ndarray:
    """[..., 32, D] codes with [..., 32, D/GROUP] scale/zero -> fp64 values."""
    rep = codes.shape[-1] // s.shape[-1]
    s64 = np.repeat(s.astype(np.float64), rep, axis=-1)
    z64 = np.repeat(z.astype(np.float64), rep, axis=-1)
    return codes.astype(np.float64) * s64 + z64


class KiviCache:
    """KIVI cache of one layer: [B, Hkv] streams of D = 128 channels.

    Blocks are kept as lists of arrays over all streams:
      k_codes [B, Hkv, n, 32, D] u8, k_scale/k_zero [B, Hkv, n, D] fp16
      v_codes [B, Hkv, n, 32, D] u8, v_scale/v_zero [B, Hkv, n, 32, D/32] fp16
      window_k, window_v [B, Hkv, w, D] fp16 with w = length % 32.
    """

    def __init__(self, B: int, Hkv: int, D: int = 128, bits: int = BITS):
        self.B, self.Hkv, self.D, self.bits = B, Hkv, D, bits
        z = lambda *s, dt: np.zeros((B, Hkv, *s), dtype=dt)  # noqa: E731
        self.k_codes = z(0, BLOCK, D, dt=np.uint8)
        self.k_scale = z(0, D, dt=np.float16)
        self.k_zero = z(0, D, dt=np.float16)
        self.v_codes = z(0, BLOCK, D, dt=np.uint8)
        self.v_scale = z(0, BLOCK, D // GROUP, dt=np.float16)
        self.v_zero = z(0, BLOCK, D // GROUP, dt=np.float16)
        self.window_k = z(0, D, dt=np.float16)
        self.window_v = z(0, D, dt=np.float16)

    @property
    def n_blocks(self) -> int:
        return self.k_codes.shape[2]

    @property
    def length(self) -> int:
        return self.n_blocks * BLOCK + self.window_k.shape[2]

    def append(self, k: np.ndarray, v: np.ndarray) -> None:
        """Append tokens k, v of [B, Hkv, T, D] (fp16)."""
        k = np.asarray(k, dtype=np.float16)
        v = np.asarray(v, dtype=np.float16)
        wk = np.concatenate([self.window_k, k], axis=2)
        wv = np.concatenate([self.window_v, v], axis=2)
        n_new = wk.shape[2] // BLOCK
        if n_new:
            B, H, D = self.B, self.Hkv, self.D
            full_k = wk[:, :, :n_new * BLOCK].astype(np.float32).reshape(B * H * n_new, BLOCK, D)
            full_v = wv[:, :, :n_new * BLOCK].astype(np.float32).reshape(B * H * n_new, BLOCK, D)
            kc, ks, kz = quantize_keys(full_k, self.bits)
            vc, vs, vz = quantize_values(full_v, self.bits)
            cat = lambda a, b: np.concatenate([a, b.reshape(B, H, n_new, *b.shape[1:])], axis=2)  # noqa: E731
            self.k_codes, self.k_scale, self.k_zero = cat(self.k_codes, kc), cat(self.k_scale, ks), cat(self.k_zero, kz)
            self.v_codes, self.v_scale, self.v_zero = cat(self.v_codes, vc), cat(self.v_scale, vs), cat(self.v_zero, vz)
        self.window_k = wk[:, :, n_new * BLOCK:].copy()
        self.window_v = wv[:, :, n_new * BLOCK:].copy()

    def keys(self) -> np.ndarray:
        """Dequantized keys [B, Hkv, S, D] fp64 (window rows exact)."""
        blk = dequantize_keys(self.k_codes, self.k_scale, self.k_zero)
        blk = blk.reshape(self.B, self.Hkv, -1, self.D)
        return np.concatenate([blk, self.window_k.astype(np.float64)], axis=2)

    def values(self) -> np.ndarray:
        """Dequantized values [B, Hkv, S, D] fp64 (window rows exact)."""
        blk = dequantize_values(self.v_codes, self.v_scale, self.v_zero)
        blk = blk.reshape(self.B, self.Hkv, -1, self.D)
        return np.concatenate([blk, self.window_v.astype(np.float64)], axis=2)

    def stored_bytes(self) -> int:
        """Bytes of codes (bits each), fp16 scale/zero and fp16 window."""
        n, w = self.n_blocks, self.window_k.shape[2]
        per_block = 2 * (BLOCK * self.D * self.bits // 8)          # K and V codes
        per_block += 2 * 2 * self.D                                 # key scale + zero per channel
        per_block += 2 * 2 * BLOCK * (self.D // GROUP)              # value scale + zero per (token, group)
        return self.B * self.Hkv * (n * per_block + 2 * w * self.D * 2)


def kivi_attend(q: np.ndarray, cache: KiviCache, scale: float | None = None) -> np.ndarray:
    """Single-token decode attention on the dequantized cache, fp64.

    q is [B, Hq, D]; returns [B, Hq, D].  Naive softmax: scores = q . K_hat /
    sqrt(D) (or `scale`), p = exp(s - max) / sum, out = p . V_hat.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Gq = Hq // cache.Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    K, V = cache.keys(), cache.values()
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            kh = h // Gq
            s = (K[b, kh] @ q[b, h]) * scale
            p = np.exp(s - s.max())
            out[b, h] = (p @ V[b, kh]) / p.sum()
    return out


# --------------------------------------------------------------------------
# Block record layout (the byte format the CUDA cache stores)
# --------------------------------------------------------------------------
#
# One record per (batch, KV head, 32-token block): the key part then the
# value part, 1536 bytes each.
#   codes: 32 tokens x 16 chunks of 8 channels, one little-endian u16 per
#          (token t, chunk c) at byte 2*(16 t + c); channel 8c + s sits at bits
#          [2k + 8h, +2) with s = 2k + h (k in 0..3, h in {0, 1}): even
#          channels of the chunk in the low byte, odd ones in the high byte,
#          each byte LSB-first [PACK].
#   key:   after the codes, fp16 scale[128] (byte 1024) then fp16 zero[128]
#          (byte 1280), one per channel.
#   value: after the codes, per (token t, channel group g of 32) an fp16
#          (scale, zero) pair at byte 1024 + 4 (4 t + g).
# The window: [batch, KV head, 2 (keys, values), 32, 128] fp16; rows
# 0 .. length % 32 - 1 are the tokens after the last complete block.

RECORD_HALF = 1536
RECORD = 2 * RECORD_HALF


def pack_codes(codes: np.ndarray) -> bytes:
    """[32, 128] codes in 0..3 -> 1024 bytes of u16 per (token, chunk)."""
    codes = np.asarray(codes, dtype=np.uint32)
    assert codes.shape == (BLOCK, 128) and codes.max(initial=0) < 4
    words = np.zeros((BLOCK, 16), dtype=np.uint32)
    for s in range(8):
        k, h = s // 2, s % 2
        words |= codes[:, s::8] << (2 * k + 8 * h)
    return words.astype("<u2").tobytes()


def pack_record(kc, ks, kz, vc, vs, vz) -> bytes:
    """One block's record from its key and value codes and fp16 scale/zero."""
    key = pack_codes(kc) + np.asarray(ks, "<f2").tobytes() + np.asarray(kz, "<f2").tobytes()
    pairs = np.stack([np.asarray(vs, "<f2"), np.asarray(vz, "<f2")], axis=-1)   # [32, 4, 2]
    val = pack_codes(vc) + pairs.tobytes()
    assert len(key) == RECORD_HALF and len(val) == RECORD_HALF
    return key + val


def records(cache: KiviCache) -> np.ndarray:
    """All records of the cache: uint8 [B, Hkv, n_blocks, 3072]."""
    out = np.zeros((cache.B, cache.Hkv, cache.n_blocks, RECORD), dtype=np.uint8)
    for b in range(cache.B):
        for h in range(cache.Hkv):
            for j in range(cache.n_blocks):
                rec = pack_record(cache.k_codes[b, h, j], cache.k_scale[b, h, j], cache.k_zero[b, h, j],
                                  cache.v_codes[b, h, j], cache.v_scale[b, h, j], cache.v_zero[b, h, j])
                out[b, h, j] = np.frombuffer(rec, dtype=np.uint8)
    return out
