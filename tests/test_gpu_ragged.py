"""Ragged per-sequence lengths on the GPU, against the ragged-lengths oracle
(oracle.ragged_oracle) and against the uniform cache.

- Equal counts through the ragged calls store exactly what the uniform calls
  store, and decode to identical outputs.
- Ragged prefill counts (shorter than a block, a whole number of blocks, and
  ragged tails), further ragged appends (zero included) and fused decode steps
  at each sequence's own position: block records bit-exact (at most 1e-5 of
  codes off by one) and fp32 tails within one ulp of the oracle's, per
  sequence; decode attention within 2e-3 of the oracle on the stored codes.
- Per-sequence rollback then re-append matches the oracle; a rollback that
  would reopen a quantized block is refused on the device (that sequence
  keeps its length, PALU_DEVERR_ROLLBACK is reported).
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle as O
from oracle import ragged_oracle as R

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATTN_TOL = 2e-3
CODE_MISMATCH_TOL = 1e-5


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _data(rng, B, H, S, r_true=20):
    A = rng.standard_normal((r_true, 128)) / math.sqrt(r_true)
    x = rng.standard_normal((B, H, S, r_true)) @ A + rng.standard_normal(128) * 0.6
    return (x + 0.05 * rng.standard_normal(x.shape)).astype(np.float16)


def _build(P, rng, B, H, cap, quantize_v=True, r=24, ng=2, S_fit=96):
    """GPU caches and their oracle twins on the same (GPU-fitted) basis."""
    caches, oracles = [], []
    for role, quant in ((P.PALU_ROLE_KEY, True), (P.PALU_ROLE_VALUE, quantize_v)):
        xf = torch.from_numpy(_data(rng, B, H, S_fit)).to(DEV)
        cfg = P.palu_config_default(n_head_groups=ng, rank=r, quantize=1 if quant else 0)
        basis, mu, _, rank, _ = P.fit(cfg, xf)
        c = P.LatentCache(cfg, role, rank, B, H, cap, basis, mu)
        Vr, mu_a = c.basis_array()
        caches.append(c)
        oracles.append(R.RaggedCache(role, Vr, mu_a, rank, B, H, cap, quant))
    return caches, oracles


def _append_ragged(P, caches, oracles, xs, counts):
    cnt = torch.tensor(counts, dtype=torch.int32, device=DEV)
    for c, o, x in zip(caches, oracles, xs):
        c.append_ragged(torch.from_numpy(x).to(DEV), cnt)
        o.append(x, counts)


def _check_storage(P, caches, oracles):
    """Per sequence: the blocks its length covers, and its tail."""
    for c, o in zip(caches, oracles):
        lens = c.lengths()
        assert lens == o.lengths, (lens, o.lengths)
        rec, tail = c.record_array(), c.tail_array()
        lay = o.seqs[0].layout
        n_codes = n_bad = 0
        for b, seq in enumerate(o.seqs):
            n = seq.length
            nb = n // 32 if seq.quantize else -(-n // 32)
            got, ref = rec[b, :, :nb], seq.blocks[0, :, :nb]
            if seq.quantize:
                cg, sg, zg = lay.unpack(got.reshape(-1, lay.record_bytes))
                co, so, zo = lay.unpack(ref.reshape(-1, lay.record_bytes))
                diff = np.abs(cg.astype(int) - co.astype(int))
                assert diff.size == 0 or diff.max() <= 1
                n_codes += diff.size
                n_bad += int((diff > 0).sum())
                assert np.array_equal(sg.view(np.uint16), so.view(np.uint16))
                assert np.array_equal(zg.view(np.uint16), zo.view(np.uint16))
                t = n % 32
                if t:
                    ga, oa = tail[b, :, :t], seq.tail[0, :, :t]
                    ulps = np.abs(ga.view(np.int32).astype(np.int64) - oa.view(np.int32).astype(np.int64))
                    assert ulps.max() <= 1
            else:
                # only the written token slots of the open block are compared
                a = lay.unpack_latents(got.reshape(-1, lay.record_bytes)).reshape(got.shape[0], nb, 32, -1)
                e = lay.unpack_latents(ref.reshape(-1, lay.record_bytes)).reshape(got.shape[0], nb, 32, -1)
                a = a.reshape(got.shape[0], nb * 32, -1)[:, :n]
                e = e.reshape(got.shape[0], nb * 32, -1)[:, :n]
                assert np.array_equal(a.view(np.uint16), e.view(np.uint16))
        assert n_bad <= CODE_MISMATCH_TOL * max(n_codes, 1)


def _oracle_attend(P, caches, q):
    """Oracle attention of each sequence over its own stored codes."""
    lens = caches[0].lengths()
    outs = []
    for b, n in enumerate(lens):
        views = []
        for c, role in zip(caches, (O.ROLE_KEY, O.ROLE_VALUE)):
            Vr, mu = c.basis_array()
            cc = c.c
            tail = c.tail_array()
            views.append(O.OracleCache.from_buffers(role, Vr, mu, cc.rank, 1, cc.kv_heads, cc.capacity,
                                                    bool(cc.quantize), c.record_array()[b:b + 1],
                                                    None if tail is None else tail[b:b + 1], n))
        outs.append(O.attend(q[b:b + 1], views[0], views[1]))
    return np.concatenate(outs, axis=0)


def _check_decode(P, caches, rng, Gq=3):
    kc, vc = caches
    B, H = kc.c.batch, kc.c.kv_heads
    q = torch.from_numpy(rng.standard_normal((B, H * Gq, 128)).astype(np.float16)).to(DEV)
    out = P.decode(kc, vc, q, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kc.sync() == 0 and vc.sync() == 0
    ref = _oracle_attend(P, caches, q.cpu().numpy())
    err = O.relative_error(out.cpu().numpy(), ref)
    assert np.isfinite(err).all() and err.max() <= ATTN_TOL, err.max()
    return q, out


@pytest.mark.parametrize("quantize_v", [True, False])
def test_equal_counts_match_the_uniform_calls(P, quantize_v):
    rng = np.random.default_rng(11)
    B, H, cap = 3, 4, 256
    (uk, uv), _ = _build(P, np.random.default_rng(5), B, H, cap, quantize_v)
    (rk, rv), _ = _build(P, np.random.default_rng(5), B, H, cap, quantize_v)
    for n in (70, 1, 33, 46):
        xk, xv = _data(rng, B, H, n), _data(rng, B, H, n)
        uk.append(torch.from_numpy(xk).to(DEV))
        uv.append(torch.from_numpy(xv).to(DEV))
        cnt = torch.full((B,), n, dtype=torch.int32, device=DEV)
        rk.append_ragged(torch.from_numpy(xk).to(DEV), cnt)
        rv.append_ragged(torch.from_numpy(xv).to(DEV), cnt)
    torch.cuda.synchronize()
    assert rk.lengths() == [150] * B and uk.sync() == 0
    for u, r_ in ((uk, rk), (uv, rv)):
        nb = 150 // 32 if u.c.quantize else -(-150 // 32)
        assert np.array_equal(u.record_array()[:, :, :nb], r_.record_array()[:, :, :nb])
        if u.c.quantize:
            assert np.array_equal(u.tail_array()[:, :, :150 % 32], r_.tail_array()[:, :, :150 % 32])
    q = torch.from_numpy(rng.standard_normal((B, H * 3, 128)).astype(np.float16)).to(DEV)
    a = P.decode(uk, uv, q, out_dtype=torch.float32)
    b = P.decode(rk, rv, q, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("quantize_v", [True, False])
def test_ragged_prefill_appends_and_steps_match_the_oracle(P, quantize_v):
    rng = np.random.default_rng(21)
    B, H, cap = 4, 4, 400
    caches, oracles = _build(P, rng, B, H, cap, quantize_v)
    # prefill: one sequence shorter than a block, one a whole number of
    # blocks, two with ragged tails
    T = 150
    xs = [_data(rng, B, H, T), _data(rng, B, H, T)]
    _append_ragged(P, caches, oracles, xs, [150, 5, 96, 61])
    _check_storage(P, caches, oracles)
    _check_decode(P, caches, rng)
    # more ragged appends, one count zero
    xs = [_data(rng, B, H, 40), _data(rng, B, H, 40)]
    _append_ragged(P, caches, oracles, xs, [3, 40, 0, 27])
    _check_storage(P, caches, oracles)
    _check_decode(P, caches, rng)
    # fused decode steps: every sequence appends one token at its own position
    kc, vc = caches
    for step in range(40):
        k1, v1 = _data(rng, B, H, 1), _data(rng, B, H, 1)
        q = torch.from_numpy(rng.standard_normal((B, H * 3, 128)).astype(np.float16)).to(DEV)
        out = P.decode_step(kc, vc, torch.from_numpy(k1[:, :, 0]).to(DEV).contiguous(),
                            torch.from_numpy(v1[:, :, 0]).to(DEV).contiguous(), q)
        oracles[0].append(k1, [1] * B)
        oracles[1].append(v1, [1] * B)
        if step in (0, 12, 39):
            torch.cuda.synchronize()
            assert kc.sync() == 0 and vc.sync() == 0
            ref = _oracle_attend(P, caches, q.cpu().numpy())
            err = O.relative_error(out.cpu().numpy(), ref)
            assert np.isfinite(err).all() and err.max() <= ATTN_TOL, (step, err.max())
    _check_storage(P, caches, oracles)


def test_ragged_rollback_then_reappend(P):
    rng = np.random.default_rng(31)
    B, H, cap = 3, 2, 300
    caches, oracles = _build(P, rng, B, H, cap, True)
    xs = [_data(rng, B, H, 120), _data(rng, B, H, 120)]
    _append_ragged(P, caches, oracles, xs, [120, 70, 45])
    # allowed: to a block boundary, inside the open block, unchanged
    lengths = [96, 66, 45]
    for c, o in zip(caches, oracles):
        c.truncate_ragged(torch.tensor(lengths, dtype=torch.int64, device=DEV))
        o.truncate(lengths)
    torch.cuda.synchronize()
    assert caches[0].sync() == 0 and caches[0].lengths() == lengths
    xs = [_data(rng, B, H, 50), _data(rng, B, H, 50)]
    _append_ragged(P, caches, oracles, xs, [50, 9, 31])
    _check_storage(P, caches, oracles)
    _check_decode(P, caches, rng)
    # refused: a length inside a quantized block (sequence 0), and growth (sequence 2)
    kc = caches[0]
    before = kc.lengths()
    bad = [before[0] - 20, before[1], before[2] + 1]
    kc.truncate_ragged(torch.tensor(bad, dtype=torch.int64, device=DEV))
    bits = ctypes.c_uint32()
    st = P.lib().palu_cache_sync(ctypes.byref(kc.c), ctypes.byref(bits),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 6 and bits.value == P.PALU_DEVERR_ROLLBACK
    assert kc.lengths() == before
