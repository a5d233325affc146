"""SVDq keys-only cache on the GPU (include/svdq.h) against its oracle
(oracle.svdq_oracle), through the C ABI.

- Per-head fit (palu_fit with one head per group) at the energy threshold
  0.95: per-head ranks, each head its own basis and mean.
- Block records: codes, fp16 scales and zeros of every stored block equal the
  oracle's encode on the GPU's bases (at most 1e-5 of codes off by one), the
  schedule's dropped channels absent; fp32 tails within one ulp.  Appends of
  several sizes (one token included) store what one long append stores.
- Decode attention within 2e-3 (max-abs over the output's L2 norm) of the
  oracle's fp64 attention on the same stored codes, with fp16 values, for
  GQA 1, 3 and 7, flat and peaked queries, explicit ranks that the schedule's
  length does not divide, and rank 1.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from oracle import svdq_oracle as S

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


def _keys(rng, B, H, S_, ranks_true=(6, 14, 24, 40), noise=0.05):
    x = np.zeros((B, H, S_, 128))
    for h in range(H):
        r = ranks_true[h % len(ranks_true)]
        A = rng.standard_normal((r, 128)) * np.linspace(2.5, 0.5, r)[:, None] / math.sqrt(r)
        x[:, h] = rng.standard_normal((B, S_, r)) @ A + rng.standard_normal(128) * 0.6
    x += noise * rng.standard_normal(x.shape)
    return x.astype(np.float16)


def _build(P, rng, B, H, cap, S_fit=160, rank=0):
    xf = torch.from_numpy(_keys(rng, B, H, S_fit)).to(DEV)
    cfg = P.palu_config_default(n_head_groups=H, rank=rank, energy_threshold=S.ENERGY_THRESHOLD)
    basis, mu, _, _, group_ranks = P.fit(cfg, xf)
    ranks = [rank] * H if rank else list(group_ranks)
    c = P.SvdqCache(B, H, ranks, cap, basis, mu)
    bases = [basis[h, :, :ranks[h]].cpu().numpy().astype(np.float32) for h in range(H)]
    oracle = S.SvdqKeyCache(bases, mu.cpu().numpy().astype(np.float32), B)
    return c, oracle


def _append(c, oracle, x):
    c.append(torch.from_numpy(x).to(DEV).contiguous())
    oracle.append(x)


def _gpu_view(c, oracle):
    """An oracle cache holding the GPU's stored codes, scales, zeros and tails."""
    torch.cuda.synchronize()
    assert c.sync() == 0
    n = c.length
    nf, nt = n // 32, n % 32
    rec, tail = c.record_array(), c.tail_array()
    view = S.SvdqKeyCache(oracle.bases, oracle.mus, oracle.B)
    for h, r in enumerate(oracle.ranks):
        codes = np.zeros((oracle.B, nf, 32, r), np.uint8)
        sc = np.zeros((oracle.B, nf, r), np.float16)
        ze = np.zeros((oracle.B, nf, r), np.float16)
        for b in range(oracle.B):
            for k in range(nf):
                codes[b, k], sc[b, k], ze[b, k] = S.unpack_record(rec[b, h, k], r)
        view.codes[h], view.scale[h], view.zero[h] = codes, sc, ze
        view.tail[h] = tail[:, h, :nt, :r].copy()
    return view


def _check_storage(c, oracle):
    view = _gpu_view(c, oracle)
    assert view.length == oracle.length == c.length
    n_codes = n_bad = 0
    for h in range(oracle.H):
        diff = np.abs(view.codes[h].astype(int) - oracle.codes[h].astype(int))
        assert diff.size == 0 or diff.max() <= 1
        n_codes += diff.size
        n_bad += int((diff > 0).sum())
        assert np.array_equal(view.scale[h].view(np.uint16), oracle.scale[h].view(np.uint16))
        assert np.array_equal(view.zero[h].view(np.uint16), oracle.zero[h].view(np.uint16))
        ulps = np.abs(view.tail[h].view(np.int32).astype(np.int64) - oracle.tail[h].view(np.int32).astype(np.int64))
        assert ulps.size == 0 or ulps.max() <= 1
    assert n_bad <= CODE_MISMATCH_TOL * max(n_codes, 1)
    return view


def _check_decode(c, oracle, rng, v, Gq, peaked=False):
    B, H = oracle.B, oracle.H
    q = rng.standard_normal((B, H * Gq, 128))
    if peaked:
        # q = 8 k_t for a cached token t of each query head's KV head
        K = oracle.keys()
        for b in range(B):
            for hq in range(H * Gq):
                q[b, hq] = 8 * K[b, hq // Gq, rng.integers(oracle.length)] / math.sqrt(128)
    q = q.astype(np.float16)
    out = c.decode(v, torch.from_numpy(q).to(DEV), out_dtype=torch.float32)
    view = _gpu_view(c, oracle)
    ref = S.svdq_attend(q, view, v[:, :, :oracle.length].cpu().numpy())
    err = O.relative_error(out.cpu().numpy(), ref)
    assert np.isfinite(err).all() and err.max() <= ATTN_TOL, err.max()


def test_svdq_records_and_appends_match_the_oracle(P):
    rng = np.random.default_rng(101)
    B, H, cap = 2, 4, 320
    c, oracle = _build(P, rng, B, H, cap)
    assert len(set(c.ranks)) > 1                      # heads land at their own ranks
    for T in (150, 1, 1, 40, 7, 33):
        _append(c, oracle, _keys(rng, B, H, T))
    _check_storage(c, oracle)


@pytest.mark.parametrize("Gq", [1, 3, 7])
def test_svdq_decode_matches_the_oracle(P, Gq):
    rng = np.random.default_rng(200 + Gq)
    B, H, cap = 2, 4, 512
    c, oracle = _build(P, rng, B, H, cap)
    _append(c, oracle, _keys(rng, B, H, 300))
    v = torch.from_numpy(rng.standard_normal((B, H, cap, 128)).astype(np.float16)).to(DEV)
    _check_decode(c, oracle, rng, v, Gq)
    _check_decode(c, oracle, rng, v, Gq, peaked=True)
    _append(c, oracle, _keys(rng, B, H, 5))         # a tail of 17 tokens
    _check_decode(c, oracle, rng, v, Gq)


@pytest.mark.parametrize("rank", [1, 8, 27, 74])
def test_svdq_explicit_ranks(P, rank):
    rng = np.random.default_rng(300 + rank)
    B, H, cap = 1, 2, 200
    c, oracle = _build(P, rng, B, H, cap, rank=rank)
    assert c.ranks == [rank] * H
    _append(c, oracle, _keys(rng, B, H, 97))
    _check_storage(c, oracle)
    v = torch.from_numpy(rng.standard_normal((B, H, cap, 128)).astype(np.float16)).to(DEV)
    _check_decode(c, oracle, rng, v, 4, peaked=True)


def test_svdq_errors(P):
    """Refusals: an append past the capacity (nothing written), a decode of an
    empty cache, query heads that are not a multiple of the KV heads or more
    than 8 per KV head, a value buffer shorter than the cache."""
    rng = np.random.default_rng(400)
    B, H, cap = 1, 2, 64
    c, oracle = _build(P, rng, B, H, cap)
    v = torch.zeros(B, H, cap, 128, dtype=torch.float16, device=DEV)
    q = torch.zeros(B, 2 * H, 128, dtype=torch.float16, device=DEV)
    with pytest.raises(P.PaluError):
        c.decode(v, q)                                         # empty
    _append(c, oracle, _keys(rng, B, H, 40))
    with pytest.raises(P.PaluError) as e:
        c.append(torch.from_numpy(_keys(rng, B, H, 25)).to(DEV))   # 65 > 64
    assert e.value.status == 3  # PALU_ERR_CAPACITY
    assert c.sync() == 0 and c.length == 40
    with pytest.raises(P.PaluError):
        c.decode(v, torch.zeros(B, 3, 128, dtype=torch.float16, device=DEV))
    with pytest.raises(P.PaluError):
        c.decode(v, torch.zeros(B, 9 * H, 128, dtype=torch.float16, device=DEV))
    with pytest.raises(P.PaluError):
        c.decode(v[:, :, :32].contiguous(), q)
    _check_storage(c, oracle)                                  # the refused calls changed nothing
