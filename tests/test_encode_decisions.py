"""The facts the prefill encoder's decisions rest on, checked on the CPU
against the oracle's quantizer (no GPU).

The encoder knows each new latent only to within a bound e, and stores a
value without the exact latent when every latent in [v - e, v + e] gives the
same stored value:

- the fp16 zero (the block minimum, rounded) and fp16 scale (max - min over
  2^b - 1 in fp32, rounded) are monotone in the minimum and maximum, so the
  two ends of their intervals bound every value in between;
- the code round((L - z) / s) is non-decreasing in L;
- the code is decided from u = (v - z) * (1/s)~, with 1/s from an approximate
  reciprocal, when |u - rint(u)| + e (1/s)~ + |u| 2^-18 + 2^-20 < 0.5: then
  every L of the interval has the oracle's code rint(u), clamped.
"""
import numpy as np

import oracle as O

F32 = np.float32


def _scale16(mx, mn, qmax):
    return (((F32(mx) - F32(mn)) / F32(qmax)).astype(F32)).astype(np.float16)


def _codes_against(s16, z16, L, qmax_bits):
    """The oracle's codes of latents L for a block whose stored scale and zero
    are (s16, z16): a block holding the minimum z and maximum z + s (2^b - 1),
    whose fp16 rounding gives back (s16, z16), and the latents under test."""
    n_hi = 1 if qmax_bits == 4 else 0
    out = []
    for chunk in np.array_split(L, max(1, len(L) // 30)):
        blk = np.empty((1, O.BLOCK, 1), F32)
        blk[0, :, 0] = chunk[0]
        blk[0, 0, 0] = F32(z16)
        qmax = 2 ** qmax_bits - 1
        blk[0, 1, 0] = F32(F32(z16) + F32(s16) * F32(qmax))
        blk[0, 2:2 + len(chunk), 0] = chunk
        codes, s_h, z_h = O.quantize_blocks(blk, n_hi)
        if s_h[0, 0] != s16 or z_h[0, 0] != z16:
            continue
        out.append((chunk, codes[0, 2:2 + len(chunk), 0]))
    return out


def test_stored_zero_and_scale_are_monotone():
    rng = np.random.default_rng(1)
    for qmax in (15, 3):
        for _ in range(4000):
            mag = 10.0 ** rng.uniform(-6, 3)
            mn = F32(rng.standard_normal() * mag)
            mx = F32(mn + abs(rng.standard_normal()) * mag * rng.uniform(0.01, 4))
            d_mn = F32(abs(rng.standard_normal()) * mag * 10.0 ** rng.uniform(-7, -1))
            d_mx = F32(abs(rng.standard_normal()) * mag * 10.0 ** rng.uniform(-7, -1))
            s0 = np.float32(_scale16(mx, mn, qmax))
            assert np.float32(_scale16(F32(mx + d_mx), mn, qmax)) >= s0
            assert np.float32(_scale16(mx, F32(mn + d_mn), qmax)) <= s0
            assert np.float32(np.float16(F32(mn + d_mn))) >= np.float32(np.float16(mn))
            # equal fp16 values at both ends of an interval fix every value inside
            lo, hi = F32(mn - d_mn), F32(mn + d_mn)
            if np.float16(lo) == np.float16(hi):
                for t in rng.uniform(0, 1, 5):
                    assert np.float16(F32(lo + F32(t) * (hi - lo))) == np.float16(lo)


def test_codes_are_non_decreasing_in_the_latent():
    rng = np.random.default_rng(2)
    for bits in (4, 2):
        for _ in range(60):
            z16 = np.float16(rng.standard_normal())
            s16 = np.float16(abs(rng.standard_normal()) * 0.3 + 1e-3)
            qmax = 2 ** bits - 1
            L = np.sort(F32(z16) + F32(s16) * rng.uniform(-0.5, qmax + 0.5, 300).astype(F32)).astype(F32)
            for chunk, codes in _codes_against(s16, z16, L, bits):
                assert np.all(np.diff(codes.astype(int)) >= 0)


def test_interval_code_decision_matches_the_oracle():
    """The decision rule with a reciprocal off by up to 2^-22 relative: when
    it claims a code, every latent of the interval has that code."""
    rng = np.random.default_rng(3)
    claimed = 0
    for bits in (4, 2):
        qmax = 2 ** bits - 1
        for _ in range(300):
            z16 = np.float16(rng.standard_normal())
            s16 = np.float16(abs(rng.standard_normal()) * 0.3 + 1e-3)
            s32, z32 = F32(s16), F32(z16)
            inv = F32(F32(1.0) / s32 * F32(1.0 + rng.uniform(-1, 1) * 2.0 ** -22))
            v = (z32 + s32 * rng.uniform(-0.6, qmax + 0.6, 64).astype(F32)).astype(F32)
            e = (np.abs(v) * F32(10.0 ** rng.uniform(-7, -3))).astype(F32)
            u = ((v - z32) * inv).astype(F32)
            du = (e * inv + np.abs(u) * F32(2.0 ** -18) + F32(2.0 ** -20)).astype(F32)
            k = np.rint(u)
            ok = np.abs(u - k) + du < 0.5
            want = np.clip(k, 0, qmax)
            for i in np.nonzero(ok)[0]:
                pts = np.array([v[i] - e[i], v[i] + e[i], v[i]] + list(v[i] + e[i] * rng.uniform(-1, 1, 4)), F32)
                pts = pts[(pts >= v[i] - e[i]) & (pts <= v[i] + e[i])]
                for chunk, codes in _codes_against(s16, z16, pts, bits):
                    assert np.all(codes == want[i]), (v[i], e[i], codes, want[i])
                    claimed += len(chunk)
    assert claimed > 1000
