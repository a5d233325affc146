"""Pins for the ragged-lengths oracle (oracle.ragged_oracle), each against
something other than itself: the pinned uniform-length cache when every
sequence has the same length, torch's SDPA with a padding mask, and the
invariants of empty appends and of rollback followed by re-append."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import ragged_oracle as R

D = 128


def _data(rng, B, H, S, r_true=20):
    A = rng.standard_normal((r_true, D)) / np.sqrt(r_true)
    x = rng.standard_normal((B, H, S, r_true)) @ A + rng.standard_normal(D) * 0.5
    return (x + 0.05 * rng.standard_normal(x.shape)).astype(np.float16)


def _caches(xk, xv, B, H, cap, r=24, ng=2, quantize_v=True):
    out = []
    for role, x, q in ((O.ROLE_KEY, xk, True), (O.ROLE_VALUE, xv, quantize_v)):
        f = O.fit(x.astype(np.float64), ng, rank=r)
        out.append(R.RaggedCache(role, f.basis.astype(np.float32), f.mu.astype(np.float32), r, B, H, cap, q))
    return out


def _valid_storage(seq):
    """The part of a sequence's storage its length makes meaningful."""
    n = seq.length
    nb = n // 32 if seq.quantize else -(-n // 32)
    return seq.blocks[:, :, :nb].copy(), seq.tail[:, :, :n % 32].copy()


@pytest.mark.parametrize("quantize_v", [True, False])
def test_equal_counts_match_the_uniform_cache(quantize_v):
    rng = np.random.default_rng(0)
    B, H, S = 3, 4, 150
    xk, xv = _data(rng, B, H, S), _data(rng, B, H, S)
    kc, vc = _caches(xk, xv, B, H, S, quantize_v=quantize_v)
    uk = O.OracleCache(O.ROLE_KEY, kc.seqs[0].V, kc.seqs[0].mu, 24, B, H, S)
    uv = O.OracleCache(O.ROLE_VALUE, vc.seqs[0].V, vc.seqs[0].mu, 24, B, H, S, quantize_v)
    t = 0
    for n in (70, 1, 33, 46):
        kc.append(xk[:, :, t:t + n], [n] * B)
        vc.append(xv[:, :, t:t + n], [n] * B)
        uk.append(xk[:, :, t:t + n])
        uv.append(xv[:, :, t:t + n])
        t += n
    assert kc.lengths == [S] * B
    for b in range(B):
        for rc, u in ((kc, uk), (vc, uv)):
            blocks, tail = _valid_storage(rc.seqs[b])
            assert np.array_equal(blocks[0], u.blocks[b, :, :blocks.shape[2]])
            assert np.array_equal(tail[0], u.tail[b, :, :tail.shape[2]])
    q = rng.standard_normal((B, H * 3, D)).astype(np.float16)
    assert np.array_equal(R.attend_ragged(q, kc, vc), O.attend(q, uk, uv))


def test_attention_matches_sdpa_with_a_padding_mask():
    """Each sequence attends over its own tokens only: torch SDPA over the
    reconstructions padded to the longest sequence, with a boolean mask."""
    rng = np.random.default_rng(1)
    B, H, Gq = 4, 2, 3
    lengths = [5, 40, 64, 97]
    S = max(lengths)
    xk, xv = _data(rng, B, H, S), _data(rng, B, H, S)
    kc, vc = _caches(xk, xv, B, H, S)
    kc.append(xk, lengths)
    vc.append(xv, lengths)
    assert kc.lengths == lengths
    K = np.zeros((B, H, S, D))
    V = np.zeros((B, H, S, D))
    for b in range(B):
        for h in range(H):
            K[b, h, :lengths[b]] = kc.seqs[b].reconstruct(0, h)
            V[b, h, :lengths[b]] = vc.seqs[b].reconstruct(0, h)
    mask = torch.from_numpy(np.arange(S)[None, :] < np.array(lengths)[:, None])[:, None, None, :]
    q = rng.standard_normal((B, H * Gq, D)).astype(np.float16)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[:, :, None],
        torch.from_numpy(K).repeat_interleave(Gq, dim=1), torch.from_numpy(V).repeat_interleave(Gq, dim=1),
        attn_mask=mask)[:, :, 0].numpy()
    assert np.allclose(R.attend_ragged(q, kc, vc), ref, rtol=1e-12, atol=1e-13)


def test_zero_count_appends_leave_a_sequence_unchanged():
    rng = np.random.default_rng(2)
    B, H, S = 3, 2, 80
    xk, xv = _data(rng, B, H, S), _data(rng, B, H, S)
    kc, _ = _caches(xk, xv, B, H, 2 * S)
    kc.append(xk[:, :, :40], [40, 17, 0])
    before = [_valid_storage(s) for s in kc.seqs]
    kc.append(xk[:, :, 40:], [0, 25, 0])
    assert kc.lengths == [40, 42, 0]
    for b in (0, 2):
        after = _valid_storage(kc.seqs[b])
        assert all(np.array_equal(a, c) for a, c in zip(before[b], after))


@pytest.mark.parametrize("back_to", [66, 64, 32, 0])
def test_rollback_then_reappend_equals_never_appending(back_to):
    """Roll sequence 1 back (inside its partial block, or to a block boundary),
    append other tokens: the same storage and attention as a cache that only
    ever saw the kept prefix and the new tokens."""
    rng = np.random.default_rng(3)
    B, H = 2, 2
    xk, xv = _data(rng, B, H, 70), _data(rng, B, H, 70)
    nk, nv = _data(rng, B, H, 30), _data(rng, B, H, 30)
    kc, vc = _caches(xk, xv, B, H, 128)
    kc.append(xk, [70, 70])
    vc.append(xv, [70, 70])
    kc.truncate([70, back_to])
    vc.truncate([70, back_to])
    kc.append(nk, [0, 30])
    vc.append(nv, [0, 30])
    # the direct cache on the same basis
    dk = R.RaggedCache(O.ROLE_KEY, kc.seqs[0].V, kc.seqs[0].mu, 24, 1, H, 128)
    dv = R.RaggedCache(O.ROLE_VALUE, vc.seqs[0].V, vc.seqs[0].mu, 24, 1, H, 128)
    for c, x, n in ((dk, xk, nk), (dv, xv, nv)):
        c.append(np.concatenate([x[1:2, :, :back_to], n[1:2]], axis=2), [back_to + 30])
    for rc, d in ((kc, dk), (vc, dv)):
        assert rc.seqs[1].length == back_to + 30
        for a, c in zip(_valid_storage(rc.seqs[1]), _valid_storage(d.seqs[0])):
            assert np.array_equal(a, c)
    q = rng.standard_normal((1, H, D)).astype(np.float16)
    assert np.array_equal(O.attend(q, kc.seqs[1], vc.seqs[1]), O.attend(q, dk.seqs[0], dv.seqs[0]))


def test_rollback_refusals():
    rng = np.random.default_rng(4)
    xk = _data(rng, 2, 2, 70)
    kc, _ = _caches(xk, xk, 2, 2, 128)
    kc.append(xk, [70, 70])
    with pytest.raises(ValueError):
        kc.truncate([50, 70])      # inside the quantized block of tokens 32-63
    with pytest.raises(ValueError):
        kc.truncate([71, 70])      # longer than the sequence
    kc.truncate([64, 69])
    assert kc.lengths == [64, 69]
