"""Plain CPU restatement of the group-head low-rank latent KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).  fp64 everywhere except
the quantizer, which takes its integer decisions in fp32 exactly as the GPU
kernel does (and as the method's fp32 latents imply).

Method sources (page title, section):
  [PALU]  "PALU — True Low-Rank Latent Storage for Keys and Values",
          sections "Usage" (config fields), "How it works" (prefill steps 1-6,
          decode steps 1-3), "Effective bit-width", "Adaptation notes".
  [SVDQ]  "veloxquant_mlx.cache.svdq_cache module", "Design" (prefill steps
          1-4: SVD, mean, projection, group quantization along the token axis
          with group_size 32).
  [KIVI]  blog post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What KIVI is"
          (asymmetric min/max group quantizer).
  [PACK]  blog post "How I built VeloxQuant-MLX", section "The Bit-Packing
          Problem" (sub-byte codes packed LSB-first, 2-bit shifts 0,2,4,6).

Readings where the pages are silent are listed in the repository's design
notes; each is restated at the function that takes it.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

ENERGY_SIGMA = 0    # cumulative sum of singular values
ENERGY_SIGMA2 = 1   # cumulative sum of squared singular values (variance)
ROLE_KEY = 0
ROLE_VALUE = 1
BLOCK = 32          # tokens per quantization group [PALU "Usage": palu_group_size=32]


# --------------------------------------------------------------------------
# Basis fit  [PALU "How it works", prefill steps 1-3]
# --------------------------------------------------------------------------

def group_rows(x: np.ndarray, n_groups: int, g: int) -> np.ndarray:
    """Rows of head group g stacked along the token axis.

    x is [B, Hkv, S, D].  The Hkv heads are split into n_groups contiguous
    groups (prefill step 1); a group's heads are stacked along the token axis
    (step 2).  The fit is on the whole prefill batch, so the batch elements
    are stacked too: rows are every (batch, head-in-group, token) triple.
    """
    B, H, S, D = x.shape
    hg = H // n_groups
    return x[:, g * hg:(g + 1) * hg].reshape(-1, D)


def fit_group(rows: np.ndarray):
    """Mean, eigenvalues and right singular directions of one group's rows.

    Prefill step 2: truncated SVD of the stacked (mean-centred) rows gives the
    shared projection V_g and the mean mu_g.  The right singular vectors of
    X_c are the eigenvectors of the centred Gram matrix X_c^T X_c, whose
    eigenvalues are the squared singular values.  Returned in descending
    order; each direction's sign is fixed so its largest-magnitude entry is
    positive (the lowest index among equal magnitudes).
    """
    X = np.asarray(rows, dtype=np.float64)
    mu = X.mean(axis=0)
    Xc = X - mu
    G = Xc.T @ Xc
    lam, V = np.linalg.eigh(G)
    order = np.argsort(-lam, kind="stable")
    lam = np.maximum(lam[order], 0.0)
    V = V[:, order]
    return mu, lam, canonical_sign(V)


def canonical_sign(V: np.ndarray) -> np.ndarray:
    """Flip each column so that its largest-|.| entry is positive."""
    V = V.copy()
    idx = np.argmax(np.abs(V), axis=0)
    s = np.sign(V[idx, np.arange(V.shape[1])])
    s[s == 0] = 1.0
    return V * s


def energy_rank(lam: np.ndarray, tau: float, mode: int = ENERGY_SIGMA) -> int:
    """Smallest k with (cumulative energy of the first k directions) / total >= tau.

    [PALU "Usage"]: "retain 90% of singular value energy".  Reading: the
    energy of direction i is its singular value sigma_i = sqrt(lambda_i)
    (mode ENERGY_SIGMA, the default) or sigma_i^2 (ENERGY_SIGMA2).  The
    cumulative sums are sequential in fp64 and the total is the last one.
    The result is clamped to [1, D].
    """
    lam = np.maximum(np.asarray(lam, dtype=np.float64), 0.0)
    w = np.sqrt(lam) if mode == ENERGY_SIGMA else lam
    cum = np.cumsum(w)
    total = cum[-1]
    if not total > 0.0:
        return 1
    ok = (cum / total) >= tau
    r = int(np.argmax(ok)) + 1 if ok.any() else len(lam)
    return max(1, min(r, len(lam)))


@dataclasses.dataclass
class Fit:
    mu: np.ndarray          # [n_g, D] fp64
    lam: np.ndarray         # [n_g, D] fp64, descending
    basis: np.ndarray       # [n_g, D, D] fp64, column j = direction j
    group_ranks: list
    rank: int               # min over groups [PALU step 3]


def fit(x: np.ndarray, n_groups: int, rank: int = 0, energy_threshold: float = 0.90,
        energy_mode: int = ENERGY_SIGMA) -> Fit:
    """Fit every head group of one tensor (K or V) of one layer.

    rank > 0 is an explicit rank; rank == 0 selects it per group by the energy
    threshold.  One rank, the minimum over groups, is used for all groups
    (prefill step 3).
    """
    D = x.shape[-1]
    mus, lams, Vs, ranks = [], [], [], []
    for g in range(n_groups):
        mu, lam, V = fit_group(group_rows(x, n_groups, g))
        mus.append(mu)
        lams.append(lam)
        Vs.append(V)
        ranks.append(min(rank, D) if rank > 0 else energy_rank(lam, energy_threshold, energy_mode))
    return Fit(np.stack(mus), np.stack(lams), np.stack(Vs), ranks, min(ranks))


# --------------------------------------------------------------------------
# Projection and mixed-bit quantization  [PALU prefill steps 4-5, decode 1-2]
# --------------------------------------------------------------------------

def n_hi_channels(r: int, hi_fraction: float = 0.25) -> int:
    """Number of leading (largest singular value) channels coded at hi_bit.

    [PALU "Usage"]: top-25% latent channels by singular value at 4 bits.
    Reading: ceil(hi_fraction * r), computed in fp64 with a 1e-9 guard
    against representation error, clamped to [0, r].
    """
    return max(0, min(r, int(math.ceil(float(hi_fraction) * r - 1e-9))))


def project(x: np.ndarray, Vr: np.ndarray, mu: np.ndarray) -> np.ndarray:
    """Latents L = (x - mu_g) @ V_g, computed in fp64 and rounded once to fp32.

    x [..., D] (fp16 values), Vr [D, r], mu [D] (the stored fp32 basis/mean).
    Latents are kept in fp32 ahead of quantization.
    """
    X = np.asarray(x, dtype=np.float64) - np.asarray(mu, dtype=np.float64)
    return (X @ np.asarray(Vr, dtype=np.float64)).astype(np.float32)


def channel_bits(r: int, n_hi: int, hi_bit: int = 4, lo_bit: int = 2) -> np.ndarray:
    return np.where(np.arange(r) < n_hi, hi_bit, lo_bit).astype(np.int64)


def quantize_blocks(L: np.ndarray, n_hi: int, hi_bit: int = 4, lo_bit: int = 2):
    """Asymmetric min/max round-to-nearest quantization of latent blocks.

    L is [N, 32, r] fp32: N blocks of 32 consecutive tokens.  For every
    (block, channel) group [SVDQ step 4: groups of group_size tokens along the
    token axis; KIVI quantizer]:
        zero  = min(g),   scale = (max(g) - min(g)) / (2^b - 1)
        q     = round((g - zero) / scale)  in [0, 2^b - 1]
    with b = hi_bit for the first n_hi channels and lo_bit for the rest.
    Readings: scale and zero are stored as fp16 (round-to-nearest-even); the
    codes are computed against the stored fp16 values in fp32 IEEE arithmetic
    (no fused multiply-add), round half to even, clamped to the code range; a
    zero stored scale gives code 0 for the whole group.
    Returns codes uint8 [N, 32, r], scale fp16 [N, r], zero fp16 [N, r].
    """
    L = np.asarray(L, dtype=np.float32)
    N, T, r = L.shape
    assert T == BLOCK
    qmax = (2 ** channel_bits(r, n_hi, hi_bit, lo_bit) - 1).astype(np.float32)   # [r]
    mn = L.min(axis=1)                                        # [N, r] fp32
    mx = L.max(axis=1)
    scale = ((mx - mn) / qmax).astype(np.float32)             # fp32 subtract, fp32 divide
    s_h = scale.astype(np.float16)
    z_h = mn.astype(np.float16)
    s32 = s_h.astype(np.float32)[:, None, :]
    z32 = z_h.astype(np.float32)[:, None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((L - z32) / s32)
    q = np.where(s32 == 0, 0.0, q)
    q = np.clip(q, 0.0, qmax[None, None, :])
    return q.astype(np.uint8), s_h, z_h


def dequantize(codes: np.ndarray, s_h: np.ndarray, z_h: np.ndarray) -> np.ndarray:
    """L_hat = code * scale + zero (exact in fp64).  codes [..., 32, r], s/z [..., r]."""
    return (codes.astype(np.float64) * s_h.astype(np.float64)[..., None, :]
            + z_h.astype(np.float64)[..., None, :])


def effective_bits(r: int, D: int, n_hi: int, hi_bit: int = 4, lo_bit: int = 2) -> float:
    """Code bits per cached element of the original [S, D] tensor.

    [PALU "Effective bit-width"]: (r/D) * (0.25*4 + 0.75*2) when a quarter of
    the r channels are at 4 bits; in general (n_hi*hi_bit + (r-n_hi)*lo_bit)/D.
    Scale/zero metadata is not part of the page's formula.
    """
    return (n_hi * hi_bit + (r - n_hi) * lo_bit) / D


# --------------------------------------------------------------------------
# Block record layout
# --------------------------------------------------------------------------
#
# A block record holds one 32-token group of one (batch, KV head) stream.
# Channels are split into a hi section (first n_hi channels, 4-bit) and a lo
# section (the rest, 2-bit); each section is cut into octets of 8 channels,
# the last octet of a section padded with zero channels.  Codes are packed
# LSB-first [PACK] into little-endian units: a 4-bit octet is 32 u32 words,
# a 2-bit octet 32 u16 halfwords; lo octets are stored in pairs, the two
# halfwords of lane i side by side, with an odd last octet on its own.  The
# position of each code inside its unit follows the register fragments of a
# 16x8x16 tensor-core product, so a GPU lane finds its operands in one load:
#   lane = 4*g + c,  field k in 0..3,  half in {0, 1}
#   4-bit: bits [4k + 16*half, +4) of the u32 word of the lane
#   2-bit: bits [2k +  8*half, +2) of the u16 halfword of the lane
# Key records (score operand, tokens x channels):
#   token t  -> g = t % 8, k = 2*(t // 16) + (t % 16) // 8
#   slot s   -> c = s // 2, half = s % 2      (slot = channel within octet)
# Value records (weighted-sum operand, channels x tokens):
#   slot s   -> g = s
#   token t  -> c = (t % 8) // 2, half = t % 2, k = 2*(t // 16) + (t % 16) // 8
# After the codes: per padded channel p = 8*octet + slot, fp16 scale and zero:
#   key:   scale[p] at 2p, zero[p] at 2*n_pad + 2p    (two arrays)
#   value: scale[p] at 4p, zero[p] at 4p + 2          (interleaved pairs)
# Values kept as fp16 latents (quantize_values=False) use one record per
# 32-token block too: octets over all r channels, 512 bytes each, the fp16
# latent of (t, channel 8o+s) at 512*o + 16*lane + 4*k + 2*half with the
# value-record mapping above.

@dataclasses.dataclass(frozen=True)
class Layout:
    role: int
    r: int
    n_hi: int
    quantize: bool = True

    @property
    def n_hi_oct(self):
        return -(-self.n_hi // 8) if self.quantize else 0

    @property
    def n_lo_oct(self):
        return -(-(self.r - self.n_hi) // 8) if self.quantize else 0

    @property
    def n_oct(self):
        return self.n_hi_oct + self.n_lo_oct if self.quantize else -(-self.r // 8)

    @property
    def n_pad(self):
        return 8 * self.n_oct

    @property
    def sz_base(self):
        return 128 * self.n_hi_oct + 64 * self.n_lo_oct

    @property
    def record_bytes(self):
        if not self.quantize:
            return 512 * self.n_oct
        return self.sz_base + 4 * self.n_pad

    def padded_channel(self, j: int) -> tuple[int, int]:
        """(octet, slot) of latent channel j."""
        if not self.quantize or j < self.n_hi:
            return j // 8, j % 8
        jj = j - self.n_hi
        return self.n_hi_oct + jj // 8, jj % 8

    def lane_field(self, t: int, slot: int) -> tuple[int, int, int]:
        """(lane, field k, half) of token t, octet slot."""
        k = 2 * (t // 16) + (t % 16) // 8
        if self.role == ROLE_KEY:
            g, c, half = t % 8, slot // 2, slot % 2
        else:
            g, c, half = slot, (t % 8) // 2, t % 2
        return 4 * g + c, k, half

    def code_position(self, t: int, j: int) -> tuple[int, int, int]:
        """(byte offset in the record, bit shift within that byte, width) of code (t, j)."""
        octet, slot = self.padded_channel(j)
        lane, k, half = self.lane_field(t, slot)
        if octet < self.n_hi_oct:
            unit = 128 * octet + 4 * lane
            bit = 4 * k + 16 * half
            width = 4
        else:
            lo = octet - self.n_hi_oct
            base = 128 * self.n_hi_oct
            if lo < 2 * (self.n_lo_oct // 2):
                unit = base + 128 * (lo // 2) + 4 * lane + 2 * (lo % 2)
            else:
                unit = base + 128 * (self.n_lo_oct // 2) + 2 * lane
            bit = 2 * k + 8 * half
            width = 2
        return unit + bit // 8, bit % 8, width

    def scale_zero_offsets(self, j: int) -> tuple[int, int]:
        octet, slot = self.padded_channel(j)
        p = 8 * octet + slot
        if self.role == ROLE_KEY:
            return self.sz_base + 2 * p, self.sz_base + 2 * self.n_pad + 2 * p
        return self.sz_base + 4 * p, self.sz_base + 4 * p + 2

    def latent_offset(self, t: int, j: int) -> int:
        """Byte offset of the fp16 latent (t, j) in an unquantized value record."""
        octet, slot = j // 8, j % 8
        lane, k, half = self.lane_field(t, slot)
        return 512 * octet + 16 * lane + 4 * k + 2 * half

    # -- vectorised tables (built once per layout by looping the definitions above)
    def _tables(self):
        tab = self.__dict__.get("_tab_cache")
        if tab is None:
            T, r = BLOCK, self.r
            if self.quantize:
                byte = np.zeros((T, r), np.int64)
                shift = np.zeros((T, r), np.int64)
                for t in range(T):
                    for j in range(r):
                        byte[t, j], shift[t, j], _ = self.code_position(t, j)
                so = np.array([self.scale_zero_offsets(j)[0] for j in range(r)], np.int64)
                zo = np.array([self.scale_zero_offsets(j)[1] for j in range(r)], np.int64)
                tab = (byte, shift, so, zo)
            else:
                off = np.zeros((T, r), np.int64)
                for t in range(T):
                    for j in range(r):
                        off[t, j] = self.latent_offset(t, j)
                tab = (off,)
            object.__setattr__(self, "_tab_cache", tab)
        return tab

    def pack(self, codes: np.ndarray, s_h: np.ndarray, z_h: np.ndarray) -> np.ndarray:
        """codes [N, 32, r] uint8, s/z [N, r] fp16 -> records uint8 [N, record_bytes]."""
        byte, shift, so, zo = self._tables()
        N = codes.shape[0]
        rec = np.zeros((N, self.record_bytes), np.int64)
        vals = codes.astype(np.int64) << shift[None]
        np.add.at(rec, (np.arange(N)[:, None, None], byte[None]), vals)   # fields are disjoint
        rec = rec.astype(np.uint8)
        sb = s_h.astype(np.float16).view(np.uint8).reshape(N, self.r, 2)
        zb = z_h.astype(np.float16).view(np.uint8).reshape(N, self.r, 2)
        for b in range(2):
            rec[np.arange(N)[:, None], so[None] + b] = sb[:, :, b]
            rec[np.arange(N)[:, None], zo[None] + b] = zb[:, :, b]
        return rec

    def unpack(self, rec: np.ndarray):
        """records [N, record_bytes] -> codes [N, 32, r] uint8, s, z [N, r] fp16."""
        byte, shift, so, zo = self._tables()
        rec = np.asarray(rec, np.uint8)
        N = rec.shape[0]
        widths = channel_bits(self.r, self.n_hi, 4, 2)
        mask = (1 << widths) - 1
        codes = (rec[:, byte].astype(np.int64) >> shift[None]) & mask[None, None, :]
        s = np.stack([rec[:, so], rec[:, so + 1]], axis=-1).copy().view(np.float16)[..., 0]
        z = np.stack([rec[:, zo], rec[:, zo + 1]], axis=-1).copy().view(np.float16)[..., 0]
        return codes.astype(np.uint8), s, z

    def pack_latents(self, lat16: np.ndarray, rec: np.ndarray | None = None, tokens=None) -> np.ndarray:
        """fp16 latents [N, 32, r] -> unquantized value records (only `tokens` written)."""
        (off,) = self._tables()
        N = lat16.shape[0]
        if rec is None:
            rec = np.zeros((N, self.record_bytes), np.uint8)
        tsel = np.arange(BLOCK) if tokens is None else np.asarray(tokens)
        b = lat16.astype(np.float16).view(np.uint8).reshape(N, BLOCK, self.r, 2)
        for i in range(2):
            rec[np.arange(N)[:, None, None], off[tsel][None] + i] = b[:, tsel][..., i]
        return rec

    def unpack_latents(self, rec: np.ndarray) -> np.ndarray:
        (off,) = self._tables()
        rec = np.asarray(rec, np.uint8)
        lo = rec[:, off].astype(np.uint16)
        hi = rec[:, off + 1].astype(np.uint16)
        return (lo | (hi << 8)).view(np.float16)


# --------------------------------------------------------------------------
# The cache  [PALU "How it works"]
# --------------------------------------------------------------------------

class OracleCache:
    """Latent storage for one tensor (K or V) of one layer.

    Holds the same buffers as the GPU cache: block records
    [B, Hkv, n_blk_cap, record_bytes] and, for quantized caches, an fp32 tail
    [B, Hkv, 32, r] for the current partial block.

    Reading of the decode append (decode steps 1-2 say "quantize and append"
    but a 32-token group is incomplete when tokens arrive one at a time):
    latents accumulate unquantized in the tail; when position p completes a
    block (p % 32 == 31) that block's 32 latents are quantized exactly as a
    prefill block.  Prefill remainders go to the tail the same way, so a
    prefill of S tokens followed by n appends stores the same codes as one
    prefill of S + n tokens.  Unquantized values (quantize_values=False) are
    rounded to fp16 at append time and stored directly.
    """

    def __init__(self, role: int, basis: np.ndarray, mu: np.ndarray, r: int, B: int, Hkv: int,
                 capacity: int, quantize: bool = True, hi_fraction: float = 0.25,
                 hi_bit: int = 4, lo_bit: int = 2):
        basis = np.asarray(basis, np.float32)
        self.n_groups = basis.shape[0]
        self.V = basis[:, :, :r].copy()          # [n_g, D, r] fp32 (stored basis)
        self.mu = np.asarray(mu, np.float32).copy()
        self.role, self.r, self.B, self.Hkv, self.capacity = role, r, B, Hkv, capacity
        self.quantize = quantize
        self.n_hi = n_hi_channels(r, hi_fraction) if quantize else 0
        self.hi_bit, self.lo_bit = hi_bit, lo_bit
        self.layout = Layout(role, r, self.n_hi, quantize)
        self.n_blk_cap = -(-capacity // BLOCK)
        self.blocks = np.zeros((B, Hkv, self.n_blk_cap, self.layout.record_bytes), np.uint8)
        self.tail = np.zeros((B, Hkv, BLOCK, r), np.float32)
        self.length = 0

    def group_of(self, h: int) -> int:
        return h // (self.Hkv // self.n_groups)

    def latents_of(self, x: np.ndarray) -> np.ndarray:
        """Project new tokens x [B, Hkv, T, D] -> fp32 [B, Hkv, T, r]."""
        out = np.empty(x.shape[:3] + (self.r,), np.float32)
        for h in range(self.Hkv):
            g = self.group_of(h)
            out[:, h] = project(x[:, h], self.V[g], self.mu[g])
        return out

    def append(self, x: np.ndarray) -> None:
        x = np.asarray(x)
        B, H, T, D = x.shape
        if T == 0:
            return
        if self.length + T > self.capacity:
            raise ValueError("append beyond capacity")
        L = self.latents_of(x)
        p0, p1 = self.length, self.length + T
        for blk in range(p0 // BLOCK, (p1 - 1) // BLOCK + 1):
            lo, hi = blk * BLOCK, min(blk * BLOCK + BLOCK, p1)
            new_lo = max(lo, p0)
            if not self.quantize:
                lat = np.zeros((B * H, BLOCK, self.r), np.float16)
                lat[:, new_lo - lo:hi - lo] = L[:, :, new_lo - p0:hi - p0].reshape(B * H, -1, self.r)
                rec = self.blocks[:, :, blk].reshape(B * H, -1).copy()
                rec = self.layout.pack_latents(lat, rec, tokens=np.arange(new_lo - lo, hi - lo))
                self.blocks[:, :, blk] = rec.reshape(B, H, -1)
                continue
            # gather the block's latents: earlier ones from the tail, new ones from L
            blk_lat = self.tail.copy()
            blk_lat[:, :, new_lo - lo:hi - lo] = L[:, :, new_lo - p0:hi - p0]
            if hi - lo == BLOCK:
                codes, s, z = quantize_blocks(blk_lat.reshape(B * H, BLOCK, self.r), self.n_hi,
                                              self.hi_bit, self.lo_bit)
                self.blocks[:, :, blk] = self.layout.pack(codes, s, z).reshape(B, H, -1)
                self.tail[:] = 0.0
            else:
                self.tail[:, :, new_lo - lo:hi - lo] = L[:, :, new_lo - p0:hi - p0]
        self.length = p1

    # -- reading back
    def latents(self, b: int, h: int) -> np.ndarray:
        """fp64 latents of every cached token of stream (b, h): dequantized
        codes of full blocks, then the fp32 tail; fp16 latents if unquantized."""
        n_full = self.length // BLOCK
        n_tail = self.length % BLOCK
        if not self.quantize:
            nb = -(-self.length // BLOCK)
            lat = self.layout.unpack_latents(self.blocks[b, h, :nb]).astype(np.float64)
            return lat.reshape(-1, self.r)[: self.length]
        parts = []
        if n_full:
            codes, s, z = self.layout.unpack(self.blocks[b, h, :n_full])
            parts.append(dequantize(codes, s, z).reshape(-1, self.r))
        if n_tail:
            parts.append(self.tail[b, h, :n_tail].astype(np.float64))
        return np.concatenate(parts, axis=0) if parts else np.zeros((0, self.r))

    def reconstruct(self, b: int, h: int) -> np.ndarray:
        """K_hat or V_hat = L_hat @ V_g^T + mu_g in fp64 [PALU prefill step 6]."""
        g = self.group_of(h)
        return self.latents(b, h) @ self.V[g].astype(np.float64).T + self.mu[g].astype(np.float64)

    @classmethod
    def from_buffers(cls, role, basis_Vr, mu, r, B, Hkv, capacity, quantize, blocks, tail, length,
                     hi_fraction=0.25):
        """A view of cache contents produced elsewhere (same layout)."""
        c = cls(role, basis_Vr, mu, r, B, Hkv, capacity, quantize, hi_fraction)
        c.blocks = np.asarray(blocks, np.uint8).reshape(c.blocks.shape).copy()
        if quantize:
            c.tail = np.asarray(tail, np.float32).reshape(c.tail.shape).copy()
        c.length = int(length)
        return c

    def stats(self):
        """Byte accounting [PALU "Evidence": compressed bytes < fp16 bytes]."""
        D = self.V.shape[1]
        n_tok = self.B * self.Hkv * self.length
        if self.quantize:
            # codes exist for full blocks only; the partial block is held unquantized
            code_bits = self.n_hi * self.hi_bit + (self.r - self.n_hi) * self.lo_bit
            code_bytes = self.B * self.Hkv * (self.length // BLOCK) * BLOCK * code_bits / 8.0
            meta_bytes = (self.length // BLOCK) * self.B * self.Hkv * self.r * 4
            tail_bytes = (self.length % BLOCK) * self.B * self.Hkv * self.r * 4
        else:
            code_bytes, meta_bytes, tail_bytes = n_tok * self.r * 2, 0, 0
        return dict(code_bytes=code_bytes, meta_bytes=meta_bytes, tail_bytes=tail_bytes,
                    fp16_bytes=n_tok * D * 2,
                    effective_bits=(effective_bits(self.r, D, self.n_hi, self.hi_bit, self.lo_bit)
                                    if self.quantize else 16.0 * self.r / D))


# --------------------------------------------------------------------------
# Decode attention  [PALU prefill step 6 / decode step 3]
# --------------------------------------------------------------------------

def attend(q: np.ndarray, kc: OracleCache, vc: OracleCache, scale: float | None = None,
           heads=None) -> np.ndarray:
    """Single-token decode attention over the reconstructed cache, in fp64.

    Keys and values are reconstructed as L_hat @ V_g^T + mu_g and a naive
    softmax attention runs over every cached token (including the token
    appended this step), scores scaled by 1/sqrt(D) unless `scale` is given.
    GQA: query head h reads KV head h // (Hq / Hkv).
    q [B, Hq, D]; `heads` optionally restricts to a list of (b, h) pairs.
    Returns fp64 [B, Hq, D] (unfilled rows are NaN when `heads` is given).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Gq = Hq // kc.Hkv
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    out = np.full((B, Hq, D), np.nan)
    want = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else list(heads)
    by_kv = {}
    for b, h in want:
        by_kv.setdefault((b, h // Gq), []).append(h)
    for (b, kv), hs in by_kv.items():
        K = kc.reconstruct(b, kv)
        V = vc.reconstruct(b, kv)
        s = (K @ q[b, hs].T) * sc                  # [S, n]
        s = s - s.max(axis=0, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=0, keepdims=True)
        out[b, hs] = (p.T @ V)
    return out


def attend_latent(q: np.ndarray, kc: OracleCache, vc: OracleCache, scale: float | None = None) -> np.ndarray:
    """The same attention evaluated in latent space (for the equality pin):
    q~ = q V_g^K, c = q . mu_g^K, scores = (L_hat^K q~ + c) * scale,
    o = softmax-weighted sum of L_hat^V, out = o V_g^V^T + mu_g^V."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Gq = Hq // kc.Hkv
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            kv = h // Gq
            gk, gv = kc.group_of(kv), vc.group_of(kv)
            qt = q[b, h] @ kc.V[gk].astype(np.float64)
            c = q[b, h] @ kc.mu[gk].astype(np.float64)
            s = (kc.latents(b, kv) @ qt + c) * sc
            p = np.exp(s - s.max())
            p /= p.sum()
            o = p @ vc.latents(b, kv)
            out[b, h] = o @ vc.V[gv].astype(np.float64).T + vc.mu[gv].astype(np.float64)
    return out


def relative_error(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max_i |out - ref| / ||ref||_2 per (b, head) vector."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(out - ref).max(axis=-1) / np.linalg.norm(ref, axis=-1)


def subspace_residual(V_ref: np.ndarray, V_test: np.ndarray) -> float:
    """||(I - V_ref V_ref^T) V_test||_F for orthonormal column sets."""
    V_ref = np.asarray(V_ref, np.float64)
    V_test = np.asarray(V_test, np.float64)
    return float(np.linalg.norm(V_test - V_ref @ (V_ref.T @ V_test)))
