"""palu_fit_batch (several tensors, one eigensolve launch) against palu_fit
on each tensor alone and against the oracle's fit, through the C ABI.

- Three tensors with different groupings and rank rules (energy threshold
  under both readings, explicit rank): bases, means and eigenvalues equal
  palu_fit's bit for bit, and so do the ranks.
- One batch of 70 tensors x 4 groups = 280 matrices (more than one
  eigensolve launch holds): every tensor equals its own palu_fit.
- One tensor of the batch against the oracle's fit (eigenvalues, leading
  subspace), the bar of the single-tensor fit test.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _keys(rng, B, H, S, rank_true=20, noise=0.05):
    A = rng.standard_normal((rank_true, 128)) * np.linspace(3.0, 0.3, rank_true)[:, None] / math.sqrt(rank_true)
    x = rng.standard_normal((B, H, S, rank_true)) @ A + rng.standard_normal(128) * 0.5
    x += noise * rng.standard_normal(x.shape)
    return torch.from_numpy(x.astype(np.float16))


def _same(P, cfgs, xs):
    got = P.fit_batch(cfgs, xs)
    for cfg, x, (basis, mu, eig, r, gr) in zip(cfgs, xs, got):
        b1, m1, e1, r1, g1 = P.fit(cfg, x)
        assert torch.equal(basis, b1) and torch.equal(mu, m1) and torch.equal(eig, e1)
        assert (r, gr) == (r1, g1)
    return got


def test_fit_batch_equals_single_fits(P):
    rng = np.random.default_rng(11)
    B, H, S = 2, 4, 600
    xs = [_keys(rng, B, H, S).to(DEV) for _ in range(3)]
    cfgs = [P.palu_config_default(n_head_groups=2, rank=0, energy_threshold=0.9),
            P.palu_config_default(n_head_groups=4, rank=0, energy_threshold=0.8, energy_mode=P.PALU_ENERGY_SIGMA2),
            P.palu_config_default(n_head_groups=1, rank=17)]
    got = _same(P, cfgs, xs)
    assert got[2][3] == 17
    # the first tensor against the oracle's fit
    f = O.fit(xs[0].cpu().numpy().astype(np.float64), 2, rank=0, energy_threshold=0.9)
    basis, mu, eig = (t.cpu().numpy() for t in got[0][:3])
    np.testing.assert_allclose(mu, f.mu, rtol=0, atol=1e-5)
    for g in range(2):
        np.testing.assert_allclose(eig[g][:16], f.lam[g][:16], rtol=1e-4, atol=1e-6 * f.lam[g][0])
        res = O.subspace_residual(f.basis[g][:, :8], basis[g][:, :8].astype(np.float64))
        assert res <= 1e-3


def test_fit_batch_over_several_launches(P):
    rng = np.random.default_rng(12)
    xs = [_keys(rng, 1, 4, 96, rank_true=12).to(DEV) for _ in range(70)]
    cfgs = [P.palu_config_default(n_head_groups=4, rank=0, energy_threshold=0.9) for _ in range(70)]
    _same(P, cfgs, xs)


def test_fit_batch_argument_errors(P):
    rng = np.random.default_rng(13)
    x = _keys(rng, 1, 4, 64).to(DEV)
    cfg = P.palu_config_default(n_head_groups=3)  # 4 heads are not a multiple of 3 groups
    with pytest.raises(P.PaluError):
        P.fit_batch([cfg], [x])


def test_fit_batch_mixes_gram_paths(P):
    """At one shape, one grouping above 64K rows per group (tensor-core Gram,
    its own chunk layout) and one below (exact Gram) in one batch, sharing the
    partial-sum area: each equals its own palu_fit.  Tensors of different
    shapes are refused by the binding before any launch."""
    rng = np.random.default_rng(14)
    xs = [_keys(rng, 2, 8, 8200).to(DEV) for _ in range(2)]
    cfgs = [P.palu_config_default(n_head_groups=1, rank=0, energy_threshold=0.9),   # 131,200 rows a group
            P.palu_config_default(n_head_groups=8, rank=24)]                        # 16,400 rows a group
    _same(P, cfgs, xs)
    _same(P, cfgs[::-1], xs[::-1])
    with pytest.raises(ValueError):
        P.fit_batch(cfgs, [xs[0], xs[1][:, :, :100].contiguous()])
