"""Pins for the KIVI-2bit oracle (oracle.kivi_oracle), each against something
other than itself: attention on exactly representable data against torch's
SDPA, hand cases for the quantization axes and the record bytes, the
quantizer's error bound, the closed-form byte count, and the append
invariant."""
import numpy as np
import pytest
import torch

from oracle import kivi_oracle as K

D = 128


def _levels(rng, n_groups, group_len):
    """Values z + c*s with s a power of two, z a multiple of 1/64, codes c in
    0..3 with both 0 and 3 present in every group: the min/max quantizer then
    reproduces them exactly (scale (3s)/3 = s, zero = z, code = c)."""
    s = 2.0 ** rng.integers(-3, 1, size=n_groups)
    z = rng.integers(-256, 256, size=n_groups) / 64.0
    c = rng.integers(0, 4, size=(n_groups, group_len))
    c[:, 0], c[:, 1] = 0, 3
    perm = rng.permuted(np.tile(np.arange(group_len), (n_groups, 1)), axis=1)
    c = np.take_along_axis(c, perm, axis=1)
    return z[:, None] + c * s[:, None]                      # [n_groups, group_len]


def _exact_kv(rng, B, H, S):
    nb = S // 32
    # keys: groups are (block, channel) over 32 tokens
    kg = _levels(rng, B * H * nb * D, 32).reshape(B, H, nb, D, 32)
    k = np.concatenate([kg.transpose(0, 1, 2, 4, 3).reshape(B, H, nb * 32, D),
                        rng.standard_normal((B, H, S - nb * 32, D))], axis=2)
    # values: groups are (token, 32 channels)
    vg = _levels(rng, B * H * nb * 32 * (D // 32), 32).reshape(B, H, nb * 32, D)
    v = np.concatenate([vg, rng.standard_normal((B, H, S - nb * 32, D))], axis=2)
    return k.astype(np.float16), v.astype(np.float16)


@pytest.mark.parametrize("B,H,Gq,S", [(1, 1, 1, 32), (2, 2, 4, 77), (1, 4, 7, 160), (2, 1, 3, 5)])
def test_exact_levels_reduce_to_sdpa(B, H, Gq, S):
    """On data the quantizer reproduces exactly, KIVI attention is exact
    attention: compare with torch's SDPA in fp64 (GQA by repeating KV heads)."""
    rng = np.random.default_rng(S * 31 + Gq)
    k, v = _exact_kv(rng, B, H, S)
    c = K.KiviCache(B, H)
    c.append(k, v)
    assert np.array_equal(c.keys(), k.astype(np.float64))
    assert np.array_equal(c.values(), v.astype(np.float64))
    q = rng.standard_normal((B, H * Gq, D))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None],
        torch.from_numpy(k.astype(np.float64)).repeat_interleave(Gq, dim=1),
        torch.from_numpy(v.astype(np.float64)).repeat_interleave(Gq, dim=1))[:, :, 0].numpy()
    assert np.allclose(K.kivi_attend(q, c), ref, rtol=1e-12, atol=1e-13)


def test_quantization_axes_hand_case():
    """Keys: one (scale, zero) per channel over the block's 32 tokens.
    Values: one per (token, 32-channel group)."""
    rng = np.random.default_rng(1)
    k = (0.1 * rng.standard_normal((1, 1, 32, D))).astype(np.float16)
    v = (0.1 * rng.standard_normal((1, 1, 32, D))).astype(np.float16)
    k[0, 0, 3, 7] = 100.0
    v[0, 0, 3, 40] = 100.0
    c = K.KiviCache(1, 1)
    c.append(k, v)
    ks, vs = c.k_scale[0, 0, 0].astype(np.float64), c.v_scale[0, 0, 0].astype(np.float64)
    assert ks.shape == (D,) and vs.shape == (32, 4)
    assert ks[7] > 30 and np.delete(ks, 7).max() < 1
    assert vs[3, 1] > 30 and np.delete(vs.ravel(), 3 * 4 + 1).max() < 1
    # the outlier is the group maximum, so it is reproduced to within rounding
    assert c.k_codes[0, 0, 0, 3, 7] == 3 and c.v_codes[0, 0, 0, 3, 40] == 3


def test_window_holds_tokens_after_the_last_block():
    rng = np.random.default_rng(2)
    for S, nb, w in ((69, 2, 5), (64, 2, 0), (31, 0, 31), (1, 0, 1)):
        k = rng.standard_normal((2, 3, S, D)).astype(np.float16)
        v = rng.standard_normal((2, 3, S, D)).astype(np.float16)
        c = K.KiviCache(2, 3)
        c.append(k, v)
        assert c.n_blocks == nb and c.length == S
        assert np.array_equal(c.window_k, k[:, :, nb * 32:]) and np.array_equal(c.window_v, v[:, :, nb * 32:])


def test_appends_equal_one_prefill():
    rng = np.random.default_rng(3)
    S = 32 * 5 + 9
    k = rng.standard_normal((2, 2, S, D)).astype(np.float16)
    v = (3 * rng.standard_normal((2, 2, S, D))).astype(np.float16)
    one = K.KiviCache(2, 2)
    one.append(k, v)
    many = K.KiviCache(2, 2)
    t = 0
    for n in (1, 7, 31, 32, 45, 1, 1, 51):
        many.append(k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
    assert t == S
    for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero", "window_k", "window_v"):
        assert np.array_equal(getattr(one, name), getattr(many, name)), name


def test_dequantization_error_bound():
    """|x_hat - x| <= s_h/2 (round to nearest) plus what the fp16 rounding of
    scale and zero can add at the clamped ends: 3|s - s_h| + |z_h - min|."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((1, 2, 96, D)) * rng.uniform(0.01, 10, (1, 2, 1, D))).astype(np.float16)
    c = K.KiviCache(1, 2)
    c.append(x, x)
    xb = x.astype(np.float64).reshape(1, 2, 3, 32, D)
    # keys: groups over tokens
    mn, mx = xb.min(axis=3), xb.max(axis=3)
    s_h, z_h = c.k_scale.astype(np.float64), c.k_zero.astype(np.float64)
    bound = 0.5 * s_h * (1 + 1e-6) + 3 * np.abs((mx - mn) / 3 - s_h) + np.abs(z_h - mn) + 1e-12
    err = np.abs(c.keys().reshape(1, 2, 3, 32, D) - xb).max(axis=3)
    assert (err <= bound).all()
    # values: groups over 32 channels
    xg = xb.reshape(1, 2, 3, 32, 4, 32)
    mn, mx = xg.min(axis=5), xg.max(axis=5)
    s_h, z_h = c.v_scale.astype(np.float64), c.v_zero.astype(np.float64)
    bound = 0.5 * s_h * (1 + 1e-6) + 3 * np.abs((mx - mn) / 3 - s_h) + np.abs(z_h - mn) + 1e-12
    err = np.abs(c.values().reshape(1, 2, 3, 32, 4, 32) - xg).max(axis=5)
    assert (err <= bound).all()


def test_stored_bytes_closed_form():
    """Per token and KV head in blocks: 2-bit K and V codes (2 * 128 * 2 / 8 =
    64 B), key scale+zero per channel per 32 tokens (2 * 2 * 128 / 32 = 16 B),
    value scale+zero per 32 channels (2 * 2 * 4 = 16 B): 96 B, i.e. 3 bits per
    element with metadata; window tokens are fp16 K and V (512 B)."""
    B, H, S = 2, 3, 32 * 4 + 7
    rng = np.random.default_rng(5)
    x = rng.standard_normal((B, H, S, D)).astype(np.float16)
    c = K.KiviCache(B, H)
    c.append(x, x)
    assert c.stored_bytes() == B * H * (128 * 96 + 7 * 512)
    assert K.RECORD == 32 * 96


def test_record_bytes_hand_positions():
    z = np.zeros((32, D), dtype=np.uint8)
    kc = z.copy()
    kc[5, 19] = 3      # chunk 2, slot 3 = (k 1, odd): bit 10 of u16 #82 -> byte 165, bits 2-3
    kc[0, 0] = 2       # chunk 0, slot 0: byte 0, bits 0-1
    kc[31, 127] = 1    # chunk 15, slot 7 = (k 3, odd): bit 14 of u16 #511 -> byte 1023, bits 6-7
    ks = np.zeros(D, np.float16)
    kz = np.zeros(D, np.float16)
    ks[9], kz[9] = 1.0, -2.0
    vc = z.copy()
    vc[2, 6] = 3       # chunk 0, slot 6 = (k 3, even): u16 #32 -> byte 1536 + 64, bits 6-7
    vs = np.zeros((32, 4), np.float16)
    vz = np.zeros((32, 4), np.float16)
    vs[1, 2], vz[1, 2] = 0.5, 4.0
    rec = np.frombuffer(K.pack_record(kc, ks, kz, vc, vs, vz), dtype=np.uint8)
    want = np.zeros(K.RECORD, dtype=np.uint8)
    want[165] = 3 << 2
    want[0] = 2
    want[1023] = 1 << 6
    want[1024 + 18:1024 + 20] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    want[1280 + 18:1280 + 20] = np.frombuffer(np.float16(-2.0).tobytes(), np.uint8)
    want[1536 + 2 * (2 * 16 + 0)] = 3 << 6
    off = 1536 + 1024 + 4 * (4 * 1 + 2)
    want[off:off + 2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    want[off + 2:off + 4] = np.frombuffer(np.float16(4.0).tobytes(), np.uint8)
    assert np.array_equal(rec, want)
