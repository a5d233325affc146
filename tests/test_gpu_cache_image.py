"""Cache save and restore (the "prompt cache" of page "add TurboQuant KV cache
compression": a prompt prefix's cache saved to host memory and reused by a
later request), through the C ABI.

A restored cache must be the saved one: the same records, tail, basis and
length, the same decode attention bit for bit, and the same results after
further appends. Images of another kind of cache, and restores into a cache
too small for the image, are refused.
"""
import numpy as np
import pytest
import torch

import oracle as O
from test_gpu_parity import ATTN_TOL, DEV, make_caches, oracle_view, rand_lowrank

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _empty_like(P, cfg, role, c, capacity):
    """A fresh cache of the same kind as c (basis and mean are placeholders)."""
    ng = c.c.n_groups
    basis = torch.zeros(ng, 128, 128, dtype=torch.float32, device=DEV)
    mu = torch.zeros(ng, 128, dtype=torch.float32, device=DEV)
    return P.LatentCache(cfg, role, c.c.rank, c.c.batch, c.c.kv_heads, capacity, basis, mu)


@pytest.mark.parametrize("S,quantize_v", [(300, True), (256, True), (95, False), (20, True)])
def test_save_restore_roundtrip(P, S, quantize_v):
    rng = np.random.default_rng(S)
    B, Hkv, Gq, extra = 2, 4, 3, 40
    xk = rand_lowrank(rng, B, Hkv, S + extra, n_groups=2)
    xv = rand_lowrank(rng, B, Hkv, S + extra, n_groups=2)
    cfg_k = P.palu_config_default(n_head_groups=2, rank=28)
    cfg_v = P.palu_config_default(n_head_groups=2, rank=36, quantize=1 if quantize_v else 0)
    kc, vc = make_caches(P, cfg_k, cfg_v, xk[:, :, :S], xv[:, :, :S], S + extra + 8)
    img_k, img_v = kc.save(), vc.save()
    torch.cuda.synchronize()
    # restore into caches with more room than the originals
    kr = _empty_like(P, cfg_k, P.PALU_ROLE_KEY, kc, S + extra + 200)
    vr = _empty_like(P, cfg_v, P.PALU_ROLE_VALUE, vc, S + extra + 200)
    kr.restore(img_k)
    vr.restore(img_v)
    torch.cuda.synchronize()
    assert kr.sync() == 0 and vr.sync() == 0
    assert kr.length == S and vr.length == S
    for a, b in ((kc, kr), (vc, vr)):
        nb = a.c.length // 32 if a.c.quantize else -(-a.c.length // 32)
        assert np.array_equal(a.record_array()[:, :, :nb], b.record_array()[:, :, :nb])
        if a.tail is not None:
            assert np.array_equal(a.tail_array(), b.tail_array())
        ba, ma = a.basis_array()
        bb, mb = b.basis_array()
        assert np.array_equal(ba, bb) and np.array_equal(ma, mb)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * Gq, 128)).astype(np.float16)).to(DEV)
    assert torch.equal(P.decode(kc, vc, q), P.decode(kr, vr, q))
    # the restored cache keeps working: further appends give the same results
    for t in range(S, S + extra, 7):
        k1 = torch.from_numpy(xk[:, :, t:t + 7].copy()).to(DEV)
        v1 = torch.from_numpy(xv[:, :, t:t + 7].copy()).to(DEV)
        for c, x in ((kc, k1), (vc, v1), (kr, k1), (vr, v1)):
            c.append(x)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * Gq, 128)).astype(np.float16)).to(DEV)
    out_a, out_b = P.decode(kc, vc, q), P.decode(kr, vr, q)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    ref = O.attend(q.cpu().numpy(), oracle_view(kr, O.ROLE_KEY), oracle_view(vr, O.ROLE_VALUE))
    err = O.relative_error(out_b.cpu().numpy(), ref)
    assert err.max() <= ATTN_TOL, f"max rel err {err.max():.3e}"


def test_restore_refuses_other_caches_and_small_capacity(P):
    rng = np.random.default_rng(5)
    B, Hkv, S = 1, 2, 200
    xk = rand_lowrank(rng, B, Hkv, S)
    cfg = P.palu_config_default(n_head_groups=1, rank=24)
    kc, vc = make_caches(P, cfg, cfg, xk, xk, S + 8)
    img = kc.save()
    torch.cuda.synchronize()
    # another rank
    other = P.LatentCache(cfg, P.PALU_ROLE_KEY, 20, B, Hkv, S + 8, torch.zeros(1, 128, 128, device=DEV),
                          torch.zeros(1, 128, device=DEV))
    with pytest.raises(P.PaluError) as e:
        other.restore(img)
    assert e.value.status == 1  # PALU_ERR_INVALID_ARG
    # another role (a value cache of the same rank)
    with pytest.raises(P.PaluError) as e:
        vc.restore(img)
    assert e.value.status == 1  # PALU_ERR_INVALID_ARG
    # too little room
    small = _empty_like(P, cfg, P.PALU_ROLE_KEY, kc, S - 1)
    with pytest.raises(P.PaluError) as e:
        small.restore(img)
    assert e.value.status == 3  # PALU_ERR_CAPACITY
    # not an image
    with pytest.raises(P.PaluError) as e:
        kc.restore(torch.zeros(img.numel(), dtype=torch.uint8))
    assert e.value.status == 1  # PALU_ERR_INVALID_ARG
    # a truncated image
    with pytest.raises(P.PaluError) as e:
        kc.restore(img[:img.numel() - 16].clone())
    assert e.value.status == 1  # PALU_ERR_INVALID_ARG


@pytest.mark.parametrize("S,quantize_v", [(95, False), (300, True)])
def test_images_are_deterministic(P, S, quantize_v):
    """Two caches built from the same prefill give byte-identical images, the
    open block's unwritten token slots included (a record is zeroed when its
    block opens)."""
    rng = np.random.default_rng(1000 + S)
    B, Hkv = 2, 4
    xk = rand_lowrank(rng, B, Hkv, S, n_groups=2)
    xv = rand_lowrank(rng, B, Hkv, S, n_groups=2)
    cfg_k = P.palu_config_default(n_head_groups=2, rank=28)
    cfg_v = P.palu_config_default(n_head_groups=2, rank=36, quantize=1 if quantize_v else 0)
    images, keep = [], []
    for i in range(2):
        # freed device memory holding a different byte pattern each time, for
        # the caches' buffers to land on
        junk = torch.full((64 << 20,), 0x11 * (i + 1) + 0x5a, dtype=torch.uint8, device=DEV)
        del junk
        kc, vc = make_caches(P, cfg_k, cfg_v, xk, xv, S + 64)
        torch.cuda.synchronize()
        images.append((kc.save(), vc.save()))
        torch.cuda.synchronize()
        keep.append((kc, vc))
    for a, b in zip(images[0], images[1]):
        assert torch.equal(a, b)
