"""Full-size parity: one layer of each of the five workloads at its real
batch, head count and prefill length, in the launch configuration the
benchmark uses.  The oracle checks sampled outputs it can compute one by one:
the fit of every group (subspace residual, ranks), sampled block records
(bit-exact codes and scale/zero against the oracle's encode on the GPU's
basis), and sampled query heads of the decode attention after decode-step
appends (2e-3 relative, on the same stored codes)."""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "llama3b", "serving", "longctx", "qwen7b"]


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def separated(lam, r, gap=1e-2):
    for k in range(r, 0, -1):
        if lam[k - 1] > 0 and (lam[k - 1] - lam[k]) / lam[k - 1] >= gap:
            return k
    return 0


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_layer(P, name):
    from rank_latent_kv_gb300 import synth
    w = synth.WORKLOADS[name]
    dev = "cuda"
    rng = np.random.default_rng(1)
    steps = 5
    caches, fits = [], []
    for tensor, role, rr in ((0, P.PALU_ROLE_KEY, w.rank_k), (1, P.PALU_ROLE_VALUE, w.rank_v)):
        x = synth.prefill(w, 0, tensor, device=dev)
        quant = tensor == 0 or w.quantize_values
        cfg = P.palu_config_default(n_head_groups=w.n_groups, rank=rr, energy_threshold=w.energy_threshold,
                                    quantize=1 if quant else 0)
        basis, mu, eig, r, gr = P.fit(cfg, x)
        # ---- fit vs oracle (every group)
        xh = x.cpu().numpy()
        f = O.fit(xh, w.n_groups, rank=rr, energy_threshold=w.energy_threshold)
        bh, muh = basis.cpu().numpy().astype(np.float64), mu.cpu().numpy()
        np.testing.assert_allclose(muh, f.mu, rtol=0, atol=2e-5)
        for g in range(w.n_groups):
            k = separated(f.lam[g], f.group_ranks[g])
            res = O.subspace_residual(f.basis[g][:, :k], bh[g][:, :k])
            print(f"{name} tensor {tensor} group {g}: r={f.group_ranks[g]} k={k} residual {res:.2e}")
            assert res <= 1e-3
        if rr == 0:
            cums = []
            for g in range(w.n_groups):
                sg = np.sqrt(f.lam[g])
                cums.append(abs(np.cumsum(sg)[f.group_ranks[g] - 1] / sg.sum() - w.energy_threshold))
            if min(cums) > 1e-6:
                assert gr == f.group_ranks and r == f.rank
        c = P.LatentCache(cfg, role, r, w.batch, w.hkv, w.prefill + steps + 8, basis, mu)
        c.append(x)
        caches.append(c)
        fits.append((xh, quant))
        del x
    kc, vc = caches
    q_all, k1, v1 = synth.decode_inputs(w, 0, 0, device=dev, n_steps=steps)
    for s in range(steps):
        kc.append(k1[s])
        vc.append(v1[s])
    out = P.decode(kc, vc, q_all[-1], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kc.sync() == 0 and vc.sync() == 0

    # ---- sampled block records vs the oracle's encode on the GPU basis
    for c, (xh, quant), role in ((kc, fits[0], O.ROLE_KEY), (vc, fits[1], O.ROLE_VALUE)):
        Vr, mu = c.basis_array()
        cc = c.c
        lay = O.Layout(role, cc.rank, cc.n_hi, quant)
        rec = c.record_array()
        nb = w.prefill // 32
        for _ in range(24):
            b, h, blk = rng.integers(w.batch), rng.integers(w.hkv), rng.integers(nb)
            g = h // (w.hkv // w.n_groups)
            lat = O.project(xh[b, h, 32 * blk:32 * blk + 32], Vr[g], mu[g])[None]
            if quant:
                codes, s_h, z_h = O.quantize_blocks(lat, cc.n_hi)
                ref = lay.pack(codes, s_h, z_h)[0]
                got = rec[b, h, blk]
                if not np.array_equal(ref, got):
                    cg, sg, zg = lay.unpack(got[None])
                    diff = np.abs(cg.astype(int) - codes.astype(int))
                    assert diff.max() <= 1 and (diff > 0).sum() <= 1, f"block {(b, h, blk)}"
            else:
                ref = lay.unpack_latents(lay.pack_latents(lat.astype(np.float16)))
                got = lay.unpack_latents(rec[b, h, blk][None])
                assert (ref.view(np.uint16) != got.view(np.uint16)).sum() <= 1

    # ---- sampled decode heads vs the oracle on the same stored codes
    views = []
    for c, role in ((kc, O.ROLE_KEY), (vc, O.ROLE_VALUE)):
        Vr, mu = c.basis_array()
        cc = c.c
        views.append(O.OracleCache.from_buffers(role, Vr, mu, cc.rank, cc.batch, cc.kv_heads, cc.capacity,
                                                bool(cc.quantize), c.record_array(), c.tail_array(), cc.length))
    heads = sorted({(int(rng.integers(w.batch)), int(rng.integers(w.hq))) for _ in range(6)} |
                   {(0, 0), (w.batch - 1, w.hq - 1)})
    ref = O.attend(q_all[-1].cpu().numpy(), views[0], views[1], heads=heads)
    got = out.cpu().numpy()
    for b, h in heads:
        err = np.abs(got[b, h] - ref[b, h]).max() / np.linalg.norm(ref[b, h])
        assert err <= 2e-3, f"{name} head {(b, h)}: {err:.2e}"
