"""Pins for the SVDq keys-only oracle (oracle.svdq_oracle), each against
something other than itself: the pages' effective-bit figures, channel
schedules and quantizer cases worked by hand, invariants of truncation and
of appends, the quantizer's error bound, per-head ranks on constructed data,
and torch's SDPA for the attention."""
import numpy as np
import pytest
import torch

from oracle import svdq_oracle as S
from tests.conftest import golden_path

D = 128


def test_effective_bits_match_the_pages():
    rows = [l.split() for l in open(golden_path("svdq_effective_bits.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 2
    for r, d, bits in rows:
        assert S.effective_bits(int(r), int(d)) == pytest.approx(float(bits), abs=0)
        # and the page's closed form (r/D) * mean(schedule)
        assert int(r) / int(d) * np.mean(S.SCHEDULE) == pytest.approx(float(bits), abs=1e-15)


def test_channel_schedule_hand_cases():
    """Equal contiguous groups, most significant first; the extra channels of
    an uneven split go to the leading groups."""
    assert S.channel_bits(16).tolist() == [8, 8, 4, 4, 2, 2, 1, 1, 1, 1, 0, 0, 0, 0, 0, 0]
    assert S.channel_bits(10).tolist() == [8, 8, 4, 4, 2, 1, 1, 0, 0, 0]
    assert S.channel_bits(8).tolist() == [8, 4, 2, 1, 1, 0, 0, 0]
    assert S.channel_bits(3).tolist() == [8, 4, 2]
    assert S.channel_bits(1).tolist() == [8]
    assert S.channel_bits(6, (4, 2)).tolist() == [4, 4, 4, 2, 2, 2]
    assert len(S.channel_bits(127)) == 127 and S.channel_bits(127)[:16].tolist() == [8] * 16


def test_quantizer_hand_cases():
    # one 32-token group per channel: channel 0 at 1 bit, 1 at 8 bits, 2 at 0 bits
    L = np.zeros((1, 32, 3), np.float32)
    L[0, :, 0] = np.where(np.arange(32) % 2, 3.0, 1.0)   # 1 bit: min 1, max 3 -> scale 2
    L[0, 5, 0] = 2.0                                       # the midpoint: code rint(0.5) = 0
    L[0, 7, 0] = 2.5                                       # 0.75 -> 1
    L[0, :, 1] = np.arange(32) * 0.5 - 4.0                # 8 bits: scale 15.5/255, zero -4
    L[0, :, 2] = 7.0                                       # 0 bits: nothing stored
    c, s, z = S.quantize_blocks(L, np.array([1, 8, 0]))
    assert c[0, :, 0].tolist() == [0 if t in (0, 2, 4, 5, 6, 8, 10, 12, 14, 16, 18, 20, 22, 24, 26, 28, 30) else 1
                                   for t in range(32)]
    assert float(s[0, 0]) == 2.0 and float(z[0, 0]) == 1.0
    assert float(z[0, 1]) == -4.0 and float(s[0, 1]) == float(np.float16(np.float32(15.5) / np.float32(255)))
    assert c[0, 0, 1] == 0 and c[0, 31, 1] == 255
    assert (c[0, :, 2] == 0).all() and float(s[0, 2]) == 0.0 and float(z[0, 2]) == 0.0
    assert (S.dequantize(c, s, z)[0, :, 2] == 0.0).all()


def test_eight_bit_grid_is_exact():
    """Latents on a 255-step grid of power-of-two step with both ends present
    come back exactly at 8 bits."""
    rng = np.random.default_rng(0)
    step = 2.0 ** rng.integers(-6, 0, size=5)
    lo = rng.integers(-64, 64, size=5) * 0.25
    k = rng.integers(0, 256, size=(3, 32, 5)).astype(np.float64)
    k[:, 0], k[:, 1] = 0, 255
    L = (lo + k * step).astype(np.float32)
    c, s, z = S.quantize_blocks(L, np.full(5, 8))
    assert np.array_equal(S.dequantize(c, s, z), L.astype(np.float64))


def _planted(rng, B, H, S_, ranks, noise=0.0):
    x = np.zeros((B, H, S_, D))
    for h, r in enumerate(ranks):
        A = rng.standard_normal((r, D)) * np.linspace(3, 1, r)[:, None]
        x[:, h] = rng.standard_normal((B, S_, r)) @ A + rng.standard_normal(D) + noise * rng.standard_normal((B, S_, D))
    return x.astype(np.float16)


def test_per_head_ranks_from_the_energy_threshold():
    """Heads of exact ranks 3, 9 and 20 land at those ranks under a threshold
    just below full energy (sigma^2 reading): one rank per head, no minimum."""
    rng = np.random.default_rng(1)
    x = _planted(rng, 2, 3, 200, (3, 9, 20))
    # fp16 rounding of x leaves a tiny noise floor: keep 1 - 1e-6 of the variance
    _, _, ranks = S.svdq_fit(x.astype(np.float64), energy_threshold=1 - 1e-6, energy_mode=1)
    assert ranks == [3, 9, 20]
    bases, mus, ranks = S.svdq_fit(x.astype(np.float64), rank=12)
    assert ranks == [12, 12, 12] and all(b.shape == (D, 12) for b in bases)


def test_truncated_channels_do_not_reach_the_keys():
    """0-bit channels read back as zero: changing the basis columns of those
    channels leaves every reconstructed key unchanged, and their codes, scales
    and zeros are all zero."""
    rng = np.random.default_rng(2)
    x = _planted(rng, 1, 2, 96, (24, 24), noise=0.05)
    bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=16)
    a = S.SvdqKeyCache(bases, mus, B=1)
    a.append(x)
    cut = int((S.channel_bits(16) > 0).sum())                   # 10 kept of 16
    other = [b.copy() for b in bases]
    for b in other:
        b[:, cut:] = rng.standard_normal((D, 16 - cut)).astype(np.float32)
    # same latents of the kept channels: build the second cache from the first's codes
    bcache = S.SvdqKeyCache(other, mus, B=1)
    bcache.codes, bcache.scale, bcache.zero, bcache.tail = a.codes, a.scale, a.zero, a.tail
    assert a.length == 96 and a.tail[0].shape[1] == 0              # three full blocks, no tail
    assert np.array_equal(a.keys(), bcache.keys())
    for h in range(2):
        assert (a.codes[h][..., cut:] == 0).all() and (a.scale[h][..., cut:] == 0).all()
        assert (a.zero[h][..., cut:] == 0).all()


def test_latent_error_bound():
    """Per kept channel and block: |L_hat - L| <= s_h/2 plus what the fp16
    rounding of scale and zero can add at the clamped ends."""
    rng = np.random.default_rng(3)
    x = _planted(rng, 2, 2, 160, (30, 30), noise=0.1)
    bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=24)
    c = S.SvdqKeyCache(bases, mus, B=2)
    c.append(x)
    for h in range(2):
        L = (x[:, h].astype(np.float64) - mus[h].astype(np.float64)) @ bases[h].astype(np.float64)
        L = L.astype(np.float32).astype(np.float64).reshape(2, 5, 32, 24)
        Lh = c.latents(h).reshape(2, 5, 32, 24)
        bits = S.channel_bits(24)
        mn, mx = L.min(axis=2), L.max(axis=2)
        qmax = np.where(bits > 0, 2.0 ** bits - 1, 1.0)
        s_h, z_h = c.scale[h].astype(np.float64), c.zero[h].astype(np.float64)
        bound = 0.5 * s_h * (1 + 1e-6) + qmax * np.abs((mx - mn) / qmax - s_h) + np.abs(z_h - mn) + 1e-9
        err = np.abs(Lh - L).max(axis=2)
        kept = bits > 0
        assert (err[..., kept] <= bound[..., kept]).all()
        assert (Lh[..., ~kept] == 0).all()


def test_appends_equal_one_prefill():
    rng = np.random.default_rng(4)
    x = _planted(rng, 2, 2, 32 * 4 + 13, (20, 12), noise=0.05)
    bases, mus, _ = S.svdq_fit(x[:, :, :100].astype(np.float64))
    one = S.SvdqKeyCache(bases, mus, B=2)
    one.append(x)
    many = S.SvdqKeyCache(bases, mus, B=2)
    t = 0
    for n in (100, 1, 1, 27, 3, 9):
        many.append(x[:, :, t:t + n])
        t += n
    assert t == x.shape[2]
    for h in range(2):
        for name in ("codes", "scale", "zero", "tail"):
            assert np.array_equal(getattr(one, name)[h], getattr(many, name)[h]), (h, name)


@pytest.mark.parametrize("fp16_keys", [False, True])
def test_attention_matches_torch_sdpa(fp16_keys):
    """Decode attention over the reconstructed keys and the fp16 values equals
    torch's SDPA on the same tensors (GQA by repeating KV heads)."""
    rng = np.random.default_rng(5)
    B, H, Gq, S_ = 2, 2, 3, 77
    x = _planted(rng, B, H, S_, (16, 16), noise=0.05)
    v = rng.standard_normal((B, H, S_, D)).astype(np.float16)
    bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=16)
    c = S.SvdqKeyCache(bases, mus, B=B)
    c.append(x)
    q = rng.standard_normal((B, H * Gq, D))
    K = torch.from_numpy(c.keys(fp16_keys)).repeat_interleave(Gq, dim=1)
    Vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(Gq, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[:, :, None], K, Vt)[:, :, 0].numpy()
    assert np.allclose(S.svdq_attend(q, c, v, fp16_keys=fp16_keys), ref, rtol=1e-12, atol=1e-13)
    if fp16_keys:
        assert np.array_equal(c.keys(True), c.keys(False).astype(np.float16).astype(np.float64))


def test_full_rank_eight_bit_keys_are_close():
    """All channels at 8 bits and rank D: the keys come back within the
    8-bit quantization error of the latents (the basis is orthonormal)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, 1, 64, D)).astype(np.float16)
    bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=D)
    c = S.SvdqKeyCache(bases, mus, B=1, schedule=(8,))
    c.append(x)
    err = np.abs(c.keys() - x.astype(np.float64)).max()
    step = float(c.scale[0].astype(np.float64).max())
    assert err <= 0.5 * step * np.sqrt(D) + 1e-5


def test_code_bytes_closed_form():
    """Full blocks only, each channel at its width: heads of rank 16 and 10
    store 32 * (32 + 28) bits per block and batch element."""
    rng = np.random.default_rng(7)
    x = _planted(rng, 3, 2, 32 * 2 + 5, (20, 20), noise=0.05)
    bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=20)
    bases = [bases[0][:, :16], bases[1][:, :10]]
    c = S.SvdqKeyCache(bases, mus, B=3)
    c.append(x)
    assert S.channel_bits(16).sum() == 32 and S.channel_bits(10).sum() == 28
    assert c.code_bytes() == 3 * 2 * 32 * (32 + 28) / 8
    assert c.assigned_avg_bits() == pytest.approx((32 + 28) / 2 / D, abs=1e-15)


def test_tail_holds_the_tokens_after_the_last_block():
    """A block is quantized when its 32nd token arrives: S tokens give S // 32
    blocks and S % 32 unquantized latents, (x - mean) V rounded once to fp32."""
    rng = np.random.default_rng(8)
    for S_ in (31, 32, 63, 65, 1):
        x = _planted(rng, 2, 1, S_, (12,), noise=0.05)
        bases, mus, _ = S.svdq_fit(x.astype(np.float64), rank=12) if S_ > 1 else \
            ([np.eye(D, 12, dtype=np.float32)], np.zeros((1, D), np.float32), [12])
        c = S.SvdqKeyCache(bases, mus, B=2)
        for t in range(S_):
            c.append(x[:, :, t:t + 1])
        nb, w = S_ // 32, S_ % 32
        assert c.codes[0].shape[1] == nb and c.tail[0].shape[1] == w and c.length == S_
        want = ((x[:, 0, nb * 32:].astype(np.float64) - mus[0].astype(np.float64))
                @ bases[0].astype(np.float64)).astype(np.float32)
        assert np.array_equal(c.tail[0], want)


def test_record_layout_hand_positions():
    """r = 8: widths 8,4,2,1,1 kept (three 0-bit channels dropped); code bytes
    32, 16, 8, 4, 4 at offsets 0, 32, 48, 56, 60; scale/zero pairs from byte
    64; 84 bytes padded to 96.  Worked by hand: token 5 of the 4-bit channel
    sits in the high nibble of byte 32 + 2; token 13 of the 2-bit channel in
    bits 2-3 of byte 48 + 3; token 9 of the first 1-bit channel in bit 1 of
    byte 56 + 1."""
    bits, kept, offs, sz_off, nbytes = S.record_layout(8)
    assert bits.tolist() == [8, 4, 2, 1, 1, 0, 0, 0] and kept == 5
    assert offs.tolist() == [0, 32, 48, 56, 60] and sz_off == 64 and nbytes == 96
    codes = np.zeros((32, 8), np.uint8)
    codes[5, 1] = 0xB
    codes[13, 2] = 0x2
    codes[9, 3] = 1
    codes[31, 0] = 0xA7
    s_h = np.arange(1, 9).astype(np.float16)
    z_h = -np.arange(1, 9).astype(np.float16)
    rec = S.pack_record(codes, s_h, z_h, 8, 96)
    assert rec[32 + 2] == 0xB0 and rec[48 + 3] == 0x08 and rec[56 + 1] == 0x02 and rec[31] == 0xA7
    assert rec[np.r_[0:31, 33, 35:48, 49:51, 52:56, 56, 58:64]].sum() == 0
    assert rec[64:68].view(np.float16).tolist() == [1.0, -1.0]       # channel 0: scale, zero
    assert rec[80:84].view(np.float16).tolist() == [5.0, -5.0]       # channel 4
    assert (rec[84:] == 0).all()


def test_record_round_trip_at_every_width():
    rng = np.random.default_rng(5)
    for r in (1, 3, 8, 10, 27, 74, 128):
        bits, kept, _, _, nbytes = S.record_layout(r)
        codes = np.zeros((32, r), np.uint8)
        for j in range(kept):
            codes[:, j] = rng.integers(0, 2 ** int(bits[j]), size=32)
        s_h = rng.standard_normal(r).astype(np.float16)
        z_h = rng.standard_normal(r).astype(np.float16)
        s_h[kept:] = 0
        z_h[kept:] = 0
        c2, s2, z2 = S.unpack_record(S.pack_record(codes, s_h, z_h, r, nbytes + 16), r)
        assert np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint16), s_h.view(np.uint16))
        assert np.array_equal(z2.view(np.uint16), z_h.view(np.uint16))
