"""Full-size parity: one layer of each of the five workloads at its real
batch, head count and prefill length, in the launch configuration the
benchmark uses.  The oracle checks sampled outputs it can compute one by one:
the fit of every group (subspace residual, ranks), 256 sampled block records
per tensor (codes and scale/zero against the oracle's encode on the GPU's
basis, with the mismatch fractions counted over all sampled values against
1e-5), and sampled query heads of the decode attention after decode-step
appends (2e-3 relative, on the same stored codes)."""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "llama3b", "serving", "longctx", "qwen7b"]
CODE_MISMATCH_TOL = 1e-5   # fraction of codes (and of scale/zero values) allowed to differ
N_SAMPLED_BLOCKS = 256     # block records sampled per tensor (all of them when there are fewer)


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

    # ---- sampled block records vs the oracle's encode on the GPU basis.
    # The bar is aggregate over every sampled code of a tensor: at most
    # CODE_MISMATCH_TOL of the codes may differ (and then by one level), and
    # at most that fraction of the fp16 scales, zeros or unquantized latents.
    for c, (xh, quant), role in ((kc, fits[0], O.ROLE_KEY), (vc, fits[1], O.ROLE_VALUE)):
        Vr, mu = c.basis_array()
        cc = c.c
        lay = O.Layout(role, cc.rank, cc.n_hi, quant)
        rec = c.record_array()
        nb = w.prefill // 32
        all_blocks = [(b, h, k) for b in range(w.batch) for h in range(w.hkv) for k in range(nb)]
        pick = rng.choice(len(all_blocks), size=min(N_SAMPLED_BLOCKS, len(all_blocks)), replace=False)
        n_codes = n_code_bad = n_sz = n_sz_bad = n_lat = n_lat_bad = 0
        max_diff = 0
        for i in pick:
            b, h, blk = all_blocks[i]
            g = h // (w.hkv // w.n_groups)
            lat = O.project(xh[b, h, 32 * blk:32 * blk + 32], Vr[g], mu[g])[None]
            got = rec[b, h, blk][None]
            if quant:
                codes, s_h, z_h = O.quantize_blocks(lat, cc.n_hi)
                cg, sg, zg = lay.unpack(got)
                diff = np.abs(cg.astype(int) - codes.astype(int))
                max_diff = max(max_diff, int(diff.max()))
                n_codes += diff.size
                n_code_bad += int((diff > 0).sum())
                n_sz += 2 * s_h.size
                n_sz_bad += int((sg.view(np.uint16) != s_h.view(np.uint16)).sum())
                n_sz_bad += int((zg.view(np.uint16) != z_h.view(np.uint16)).sum())
            else:
                ref = lay.unpack_latents(lay.pack_latents(lat.astype(np.float16)))
                gl = lay.unpack_latents(got)
                n_lat += ref.size
                n_lat_bad += int((ref.view(np.uint16) != gl.view(np.uint16)).sum())
        print(f"{name} role {role}: {len(pick)} blocks, codes {n_code_bad}/{n_codes} differ (max {max_diff}), "
              f"scale/zero {n_sz_bad}/{n_sz}, fp16 latents {n_lat_bad}/{n_lat}")
        if quant:
            assert max_diff <= 1, f"{name} role {role}: a code differs by {max_diff}"
            assert n_code_bad <= CODE_MISMATCH_TOL * n_codes, f"{name} role {role}: {n_code_bad}/{n_codes} codes differ"
            assert n_sz_bad <= CODE_MISMATCH_TOL * n_sz, f"{name} role {role}: {n_sz_bad}/{n_sz} scale/zero differ"
        else:
            assert n_lat_bad <= CODE_MISMATCH_TOL * n_lat, f"{name} role {role}: {n_lat_bad}/{n_lat} latents differ"

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
