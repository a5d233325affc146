"""GPU path vs the CPU oracle, element by element, through the C ABI.

Bars: codes and scale/zero bit-exact (at most 1e-5 of codes off by one where
an fp32 rounding differs); decode attention within 2e-3 max-abs relative to
the output's L2 norm, compared on the same stored codes; basis subspace
residual <= 1e-3 on the well-separated leading directions.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3
CODE_MISMATCH_TOL = 1e-5


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


DEV = "cuda"


def rand_lowrank(rng, B, H, S, rank_true=24, noise=0.05, mu_scale=0.7, n_groups=1, outliers=()):
    D = 128
    x = np.empty((B, H, S, D), np.float32)
    hg = H // n_groups
    for g in range(n_groups):
        A = rng.standard_normal((rank_true, D)) / math.sqrt(rank_true)
        mu = rng.standard_normal(D) * mu_scale
        for h in range(g * hg, (g + 1) * hg):
            x[:, h] = rng.standard_normal((B, S, rank_true)) @ A + mu + noise * rng.standard_normal((B, S, D))
    for c in outliers:
        x[..., c] *= 20
    return x.astype(np.float16)


def make_caches(P, cfg_k, cfg_v, xk, xv, capacity, rank_k=None, rank_v=None):
    """Fit K and V on the GPU, build caches, append the prefill."""
    B, H, S, _ = xk.shape
    out = []
    for role, cfg, x, rr in ((P.PALU_ROLE_KEY, cfg_k, xk, rank_k), (P.PALU_ROLE_VALUE, cfg_v, xv, rank_v)):
        xt = torch.from_numpy(x).to(DEV)
        basis, mu, eig, rank, gr = P.fit(cfg, xt)
        r = rank if rr is None else rr
        c = P.LatentCache(cfg, role, r, B, H, capacity, basis, mu)
        if S:
            c.append(xt)
        out.append(c)
    return out


def oracle_view(c, role):
    Vr, mu = c.basis_array()
    cc = c.c
    return O.OracleCache.from_buffers(role, Vr, mu, cc.rank, cc.batch, cc.kv_heads, cc.capacity, bool(cc.quantize),
                                      c.record_array(), c.tail_array(), cc.length)


def compare_records(gpu_rec, ora_rec, layout, what=""):
    """Bit-exact bytes, else code-level comparison within the off-by-one allowance."""
    if np.array_equal(gpu_rec, ora_rec):
        return
    flat_g = gpu_rec.reshape(-1, layout.record_bytes)
    flat_o = ora_rec.reshape(-1, layout.record_bytes)
    if not layout.quantize:
        a = layout.unpack_latents(flat_g).astype(np.float64)
        b = layout.unpack_latents(flat_o).astype(np.float64)
        bad = a != b
        assert bad.mean() <= CODE_MISMATCH_TOL, f"{what}: {bad.sum()} fp16 latents differ"
        return
    cg, sg, zg = layout.unpack(flat_g)
    co, so, zo = layout.unpack(flat_o)
    diff = np.abs(cg.astype(int) - co.astype(int))
    frac = (diff > 0).mean()
    assert diff.max() <= 1 and frac <= CODE_MISMATCH_TOL, \
        f"{what}: {int((diff > 0).sum())} codes differ (max {diff.max()}), frac {frac:.2e}"
    sz_bad = (sg.view(np.uint16) != so.view(np.uint16)) | (zg.view(np.uint16) != zo.view(np.uint16))
    assert sz_bad.mean() <= CODE_MISMATCH_TOL, f"{what}: {sz_bad.sum()} scale/zero differ"


def check_encode(P, c, role, x_chunks):
    """Replay the same appends in the oracle on the GPU's basis; compare storage."""
    cc = c.c
    Vr, mu = c.basis_array()
    o = O.OracleCache(role, Vr, mu, cc.rank, cc.batch, cc.kv_heads, cc.capacity, bool(cc.quantize))
    for x in x_chunks:
        o.append(x)
    c.sync()
    assert cc.length == o.length
    lay = O.Layout(role, cc.rank, cc.n_hi, bool(cc.quantize))
    nb = o.length // 32 if cc.quantize else -(-o.length // 32)
    compare_records(c.record_array()[:, :, :nb], o.blocks[:, :, :nb], lay, f"role {role} r {cc.rank}")
    if cc.quantize and o.length % 32:
        # unquantized fp32 latents: equal to within one ulp (both sides round
        # the same real value to fp32; a value at a rounding midpoint may differ)
        t = o.length % 32
        ga, oa = c.tail_array()[:, :, :t], o.tail[:, :, :t]
        ulps = np.abs(ga.view(np.int32).astype(np.int64) - oa.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1 and (ulps > 0).mean() <= 1e-3
    return o


# ---------------------------------------------------------------- encode

@pytest.mark.parametrize("rank", [1, 7, 8, 9, 17, 27, 32, 52, 74, 128])
def test_encode_prefill_and_appends_bit_exact(P, rank):
    rng = np.random.default_rng(rank)
    B, H, S = 2, 4, 109                      # ragged: 3 full blocks + 13-token tail
    xk = rand_lowrank(rng, B, H, S + 40, n_groups=2)
    xv = rand_lowrank(rng, B, H, S + 40, n_groups=2)
    cfg = P.palu_config_default(n_head_groups=2, rank=rank)
    kc, vc = make_caches(P, cfg, cfg, xk[:, :, :S], xv[:, :, :S], 256)
    # single-token appends across a block boundary, then a 30-token append
    chunks_k, chunks_v = [xk[:, :, :S]], [xv[:, :, :S]]
    for t in range(S, S + 10):
        kc.append(torch.from_numpy(xk[:, :, t:t + 1].copy()).to(DEV))
        vc.append(torch.from_numpy(xv[:, :, t:t + 1].copy()).to(DEV))
        chunks_k.append(xk[:, :, t:t + 1])
        chunks_v.append(xv[:, :, t:t + 1])
    kc.append(torch.from_numpy(xk[:, :, S + 10:].copy()).to(DEV))
    vc.append(torch.from_numpy(xv[:, :, S + 10:].copy()).to(DEV))
    chunks_k.append(xk[:, :, S + 10:])
    chunks_v.append(xv[:, :, S + 10:])
    check_encode(P, kc, O.ROLE_KEY, chunks_k)
    check_encode(P, vc, O.ROLE_VALUE, chunks_v)


# multi-token appends that complete the open partial block and open a new
# one in the same call (the completing CTA reads the tail rows the new
# block's tail overwrites: the two must be ordered), over many streams
def test_encode_appends_crossing_open_blocks(P):
    rng = np.random.default_rng(123)
    B, H, S = 8, 8, 20
    sizes = [5, 40, 27, 70, 3, 33, 61]
    total = S + sum(sizes)
    xk = rand_lowrank(rng, B, H, total, n_groups=2)
    xv = rand_lowrank(rng, B, H, total, n_groups=2)
    cfg = P.palu_config_default(n_head_groups=2, rank=30)
    kc, vc = make_caches(P, cfg, cfg, xk[:, :, :S], xv[:, :, :S], total + 8)
    chunks_k, chunks_v = [xk[:, :, :S]], [xv[:, :, :S]]
    t = S
    for n in sizes:
        kc.append(torch.from_numpy(xk[:, :, t:t + n].copy()).to(DEV))
        vc.append(torch.from_numpy(xv[:, :, t:t + n].copy()).to(DEV))
        chunks_k.append(xk[:, :, t:t + n])
        chunks_v.append(xv[:, :, t:t + n])
        t += n
    check_encode(P, kc, O.ROLE_KEY, chunks_k)
    check_encode(P, vc, O.ROLE_VALUE, chunks_v)


@pytest.mark.parametrize("rank", [9, 33, 74, 128])
def test_encode_blocks_that_stress_the_bound_decisions(P, rank):
    """Blocks built so that the encoder's decisions from its error bound go
    every way: tokens within 1e-4 of the group mean (latents so small that the
    bound decides neither zero, scale nor most codes: long exact work
    lists), outlier tokens (decided from the bounds alone), exact duplicate
    tokens (tied minima and maxima), one token repeated over a block (scale
    0), the fp16 rounding of the mean repeated, and an ordinary block.  The
    records must equal the oracle's on the GPU's basis."""
    rng = np.random.default_rng(700 + rank)
    B, H, S = 2, 4, 6 * 32
    base = rand_lowrank(rng, B, H, 256, n_groups=2)
    cfg = P.palu_config_default(n_head_groups=2, rank=rank)
    basis, mu, _, _, _ = P.fit(cfg, torch.from_numpy(base).to(DEV))
    mu_h = mu.cpu().numpy()
    x = np.empty((B, H, S, 128), np.float32)
    for h in range(H):
        m = mu_h[h // 2]
        blk = [slice(32 * i, 32 * i + 32) for i in range(6)]
        x[:, h, blk[0]] = m + 1e-4 * rng.standard_normal((B, 32, 128))
        x[:, h, blk[1]] = m + rng.standard_normal((B, 32, 128)) * np.where(rng.random((B, 32, 1)) < 0.1, 100.0, 1.0)
        rows = m + rng.standard_normal((B, 8, 128))
        x[:, h, blk[2]] = rows[:, rng.integers(0, 8, 32)]
        x[:, h, blk[3]] = (m + rng.standard_normal(128))[None, None, :]
        x[:, h, blk[4]] = m
        x[:, h, blk[5]] = base[:, h, :32]
    x16 = x.astype(np.float16)
    for role, orole in ((P.PALU_ROLE_KEY, O.ROLE_KEY), (P.PALU_ROLE_VALUE, O.ROLE_VALUE)):
        c = P.LatentCache(cfg, role, rank, B, H, S + 32, basis, mu)
        c.append(torch.from_numpy(x16).to(DEV))
        check_encode(P, c, orole, [x16])


@pytest.mark.parametrize("rank", [5, 32, 100])
def test_encode_fp16_value_latents(P, rank):
    rng = np.random.default_rng(100 + rank)
    B, H, S = 1, 8, 77
    xv = rand_lowrank(rng, B, H, S + 5, n_groups=4)
    cfg = P.palu_config_default(n_head_groups=4, rank=rank, quantize=0)
    xt = torch.from_numpy(xv[:, :, :S].copy()).to(DEV)
    basis, mu, _, _, _ = P.fit(cfg, xt)
    vc = P.LatentCache(cfg, P.PALU_ROLE_VALUE, rank, B, H, 128, basis, mu)
    vc.append(xt)
    for t in range(S, S + 5):
        vc.append(torch.from_numpy(xv[:, :, t:t + 1].copy()).to(DEV))
    check_encode(P, vc, O.ROLE_VALUE, [xv[:, :, :S]] + [xv[:, :, t:t + 1] for t in range(S, S + 5)])


# ---------------------------------------------------------------- decode attention

def run_decode_case(P, B, Hkv, Gq, S, rk, rv, n_groups=2, quantize_v=True, peaked=False, seed=0, steps=2):
    rng = np.random.default_rng(seed)
    xk = rand_lowrank(rng, B, Hkv, S + steps, n_groups=n_groups)
    xv = rand_lowrank(rng, B, Hkv, S + steps, n_groups=n_groups)
    cfg_k = P.palu_config_default(n_head_groups=n_groups, rank=rk)
    cfg_v = P.palu_config_default(n_head_groups=n_groups, rank=rv, quantize=1 if quantize_v else 0)
    kc, vc = make_caches(P, cfg_k, cfg_v, xk[:, :, :S], xv[:, :, :S], S + steps + 8)
    for t in range(S, S + steps):
        kc.append(torch.from_numpy(xk[:, :, t:t + 1].copy()).to(DEV))
        vc.append(torch.from_numpy(xv[:, :, t:t + 1].copy()).to(DEV))
    Hq = Hkv * Gq
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    if peaked:
        # q = 8 k_{t*} for a random cached token of each query head's KV head
        for b in range(B):
            for h in range(Hq):
                q[b, h] = 8.0 * xk[b, h // Gq, rng.integers(0, S + steps)].astype(np.float32)
    q = q.astype(np.float16)
    out = P.decode(kc, vc, torch.from_numpy(q).to(DEV), out_dtype=torch.float32)
    torch.cuda.synchronize()
    kc.sync()
    vc.sync()
    ref = O.attend(q, oracle_view(kc, O.ROLE_KEY), oracle_view(vc, O.ROLE_VALUE))
    err = O.relative_error(out.cpu().numpy(), ref)
    assert np.isfinite(err).all()
    assert err.max() <= ATTN_TOL, f"max rel err {err.max():.3e}"
    return err.max()


@pytest.mark.parametrize("Gq", [1, 2, 3, 7, 8])
def test_decode_gqa_factors(P, Gq):
    run_decode_case(P, B=2, Hkv=4, Gq=Gq, S=300, rk=32, rv=32, seed=Gq)


@pytest.mark.parametrize("rk,rv", [(1, 1), (7, 9), (27, 52), (74, 74), (128, 128), (30, 100)])
def test_decode_ranks(P, rk, rv):
    run_decode_case(P, B=1, Hkv=4, Gq=3, S=257, rk=rk, rv=rv, seed=rk + rv)


# the per-class kernels (more than 8 octets on a side; 12-warp CTAs when the
# rings fit) with 7 and 8 query heads per KV head, on streams that one CTA
# finishes and on streams split over several CTAs and merged by the last one
@pytest.mark.parametrize("Gq", [7, 8])
@pytest.mark.parametrize("B,Hkv,S,rk,rv", [(8, 8, 300, 74, 100), (1, 2, 20011, 74, 74), (2, 2, 5000, 128, 128)])
def test_decode_class_kernels_wide_gqa(P, Gq, B, Hkv, S, rk, rv):
    run_decode_case(P, B=B, Hkv=Hkv, Gq=Gq, S=S, rk=rk, rv=rv, n_groups=2, seed=Gq + S, steps=1)


def _rank_for_octets(n):
    """Smallest rank whose mixed-bit record has n octets (oracle layout)."""
    for r in range(1, 129):
        if O.Layout(O.ROLE_KEY, r, O.n_hi_channels(r)).n_oct == n:
            return r
    raise ValueError(n)


# every key octet count 1..8 (kernels specialised on the exact count) against
# a spread of value octet counts
@pytest.mark.parametrize("ko,vo", [(k, v) for k in range(1, 9) for v in (1 + (3 * k) % 8, 9 - k)])
def test_decode_exact_octet_kernels(P, ko, vo):
    rk, rv = _rank_for_octets(ko), _rank_for_octets(vo)
    run_decode_case(P, B=1, Hkv=2, Gq=4, S=200, rk=rk, rv=rv, n_groups=1, seed=10 * ko + vo, steps=1)


# contexts long enough that warps stream several two-block stages and the
# warps' ranges cross from one (batch, KV head) stream into the next
@pytest.mark.parametrize("B,Hkv,S", [(1, 8, 20011), (2, 4, 50017)])
def test_decode_multi_block_warps(P, B, Hkv, S):
    run_decode_case(P, B=B, Hkv=Hkv, Gq=3, S=S, rk=30, rv=53, n_groups=2, seed=S, steps=1)


# more streams than the decode grid has warps to spare: CTAs that cover whole
# streams (finished in place), streams split over two CTAs (a ticket picks the
# one that merges), and contexts with no full block (tails only, several CTAs)
@pytest.mark.parametrize("B,Hkv,S", [(48, 8, 100), (16, 8, 20), (64, 8, 700)])
def test_decode_many_streams(P, B, Hkv, S):
    run_decode_case(P, B=B, Hkv=Hkv, Gq=2, S=S, rk=16, rv=24, n_groups=2, seed=B + S, steps=1)


# the fused decode step (append k, append v, attend) against the separate calls
# on identical caches, and against the oracle; steps cross block boundaries
@pytest.mark.parametrize("S,rk,rv,quantize_v", [(29, 16, 24, True), (250, 30, 53, True), (95, 32, 32, False),
                                                (3000, 74, 74, True)])
def test_decode_step_matches_separate_calls(P, S, rk, rv, quantize_v):
    rng = np.random.default_rng(S + rk)
    B, Hkv, Gq, steps = 2, 4, 3, 6
    xk = rand_lowrank(rng, B, Hkv, S + steps, n_groups=2)
    xv = rand_lowrank(rng, B, Hkv, S + steps, n_groups=2)
    cfg_k = P.palu_config_default(n_head_groups=2, rank=rk)
    cfg_v = P.palu_config_default(n_head_groups=2, rank=rv, quantize=1 if quantize_v else 0)
    ka, va = make_caches(P, cfg_k, cfg_v, xk[:, :, :S], xv[:, :, :S], S + steps + 8)
    kb, vb = make_caches(P, cfg_k, cfg_v, xk[:, :, :S], xv[:, :, :S], S + steps + 8)
    for t in range(S, S + steps):
        q = torch.from_numpy(rng.standard_normal((B, Hkv * Gq, 128)).astype(np.float16)).to(DEV)
        k1 = torch.from_numpy(xk[:, :, t:t + 1].copy()).to(DEV)
        v1 = torch.from_numpy(xv[:, :, t:t + 1].copy()).to(DEV)
        ka.append(k1)
        va.append(v1)
        out_a = P.decode(ka, va, q)
        out_b = P.decode_step(kb, vb, k1, v1, q)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), f"step {t}"
    assert kb.sync() == 0 and vb.sync() == 0
    assert kb.length == S + steps and vb.length == S + steps
    nb = (S + steps) // 32
    assert np.array_equal(kb.record_array()[:, :, :nb], ka.record_array()[:, :, :nb])
    assert np.array_equal(vb.record_array()[:, :, :nb], va.record_array()[:, :, :nb])
    ref = O.attend(q.cpu().numpy(), oracle_view(kb, O.ROLE_KEY), oracle_view(vb, O.ROLE_VALUE))
    err = O.relative_error(out_b.cpu().numpy(), ref)
    assert err.max() <= ATTN_TOL, f"max rel err {err.max():.3e}"


# the step whose key token completes a block whose scales dwarf every scale
# stored before (small prefill, one very large token): the query prescale of
# the fused step must already cover that block (no fp16 overflow), with the
# same result as the separate calls
def test_decode_step_completing_block_with_large_scales(P):
    rng = np.random.default_rng(77)
    B, Hkv, Gq, S = 2, 4, 3, 63
    xk = (rand_lowrank(rng, B, Hkv, S + 1, n_groups=2).astype(np.float32) * 0.01)
    xv = (rand_lowrank(rng, B, Hkv, S + 1, n_groups=2).astype(np.float32) * 0.01)
    xk[:, :, S] = rng.standard_normal((B, Hkv, 128)) * 400.0
    xk, xv = xk.astype(np.float16), xv.astype(np.float16)
    cfg = P.palu_config_default(n_head_groups=2, rank=24)
    ka, va = make_caches(P, cfg, cfg, xk[:, :, :S], xv[:, :, :S], S + 8)
    kb, vb = make_caches(P, cfg, cfg, xk[:, :, :S], xv[:, :, :S], S + 8)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * Gq, 128)).astype(np.float16)).to(DEV)
    k1 = torch.from_numpy(xk[:, :, S:S + 1].copy()).to(DEV)
    v1 = torch.from_numpy(xv[:, :, S:S + 1].copy()).to(DEV)
    ka.append(k1)
    va.append(v1)
    out_a = P.decode(ka, va, q)
    out_b = P.decode_step(kb, vb, k1, v1, q)
    torch.cuda.synchronize()
    assert kb.sync() == 0 and vb.sync() == 0
    assert torch.isfinite(out_b).all()
    assert torch.equal(out_a, out_b)
    ref = O.attend(q.cpu().numpy(), oracle_view(kb, O.ROLE_KEY), oracle_view(vb, O.ROLE_VALUE))
    err = O.relative_error(out_b.cpu().numpy(), ref)
    assert err.max() <= ATTN_TOL, f"max rel err {err.max():.3e}"


@pytest.mark.parametrize("S", [1, 5, 31, 32, 33, 64, 95, 1000, 4099])
def test_decode_lengths(P, S):
    run_decode_case(P, B=1, Hkv=2, Gq=3, S=S, rk=16, rv=24, n_groups=1, seed=S, steps=1)


@pytest.mark.parametrize("quantize_v", [True, False])
def test_decode_peaked_attention(P, quantize_v):
    run_decode_case(P, B=2, Hkv=4, Gq=3, S=700, rk=32, rv=32, quantize_v=quantize_v, peaked=True, seed=7)


def test_decode_fp16_value_latents(P):
    run_decode_case(P, B=3, Hkv=8, Gq=3, S=513, rk=32, rv=32, n_groups=4, quantize_v=False, seed=11)


def test_decode_fp16_output_and_scale(P):
    rng = np.random.default_rng(3)
    B, H, S = 1, 2, 200
    xk = rand_lowrank(rng, B, H, S)
    xv = rand_lowrank(rng, B, H, S)
    cfg = P.palu_config_default(n_head_groups=1, rank=20)
    kc, vc = make_caches(P, cfg, cfg, xk, xv, 256)
    q = rng.standard_normal((B, 4, 128)).astype(np.float16)
    out = P.decode(kc, vc, torch.from_numpy(q).to(DEV), out_dtype=torch.float16, softmax_scale=0.05)
    ref = O.attend(q, oracle_view(kc, O.ROLE_KEY), oracle_view(vc, O.ROLE_VALUE), scale=0.05)
    assert O.relative_error(out.float().cpu().numpy(), ref).max() <= ATTN_TOL


# ---------------------------------------------------------------- fit

def leading_separated(lam, r, gap=1e-2):
    """Largest k <= r with relative gap (lam_k - lam_{k+1}) / lam_k >= gap."""
    for k in range(r, 0, -1):
        if k < len(lam) and lam[k - 1] > 0 and (lam[k - 1] - lam[k]) / lam[k - 1] >= gap:
            return k
    return 0


@pytest.mark.parametrize("kind", ["planted", "spectrum"])
def test_fit_matches_oracle(P, kind):
    from rank_latent_kv_gb300 import synth
    if kind == "planted":
        w = synth.scaled(synth.WORKLOADS["tiny"])
    else:
        w = synth.scaled(synth.WORKLOADS["llama3b"], prefill=2048)
    x = synth.prefill(w, 0, 0, device="cpu")
    cfg = P.palu_config_default(n_head_groups=w.n_groups, rank=w.rank_k,
                                energy_threshold=w.energy_threshold)
    basis, mu, eig, rank, gr = P.fit(cfg, x.to(DEV))
    f = O.fit(x.numpy().astype(np.float64), w.n_groups, rank=w.rank_k, energy_threshold=w.energy_threshold)
    basis, mu, eig = basis.cpu().numpy(), mu.cpu().numpy(), eig.cpu().numpy()
    np.testing.assert_allclose(mu, f.mu, rtol=0, atol=1e-5)
    for g in range(w.n_groups):
        lam = f.lam[g]
        np.testing.assert_allclose(eig[g][:64], lam[:64], rtol=1e-4, atol=1e-6 * lam[0])
        r = f.group_ranks[g]
        k = leading_separated(lam, r)
        assert k >= 1
        res = O.subspace_residual(f.basis[g][:, :k], basis[g][:, :k].astype(np.float64))
        print(f"group {g}: r={r} separated k={k} subspace residual {res:.3e}")
        assert res <= 1e-3
        # columns beyond the separated ones still capture the optimal energy
        G = np.einsum("ij,ik->jk", *(2 * [O.group_rows(x.numpy().astype(np.float64), w.n_groups, g) - f.mu[g]]))
        Vg = basis[g][:, :r].astype(np.float64)
        Vo = f.basis[g][:, :r]
        assert np.trace(Vg.T @ G @ Vg) >= np.trace(Vo.T @ G @ Vo) * (1 - 1e-6)
        # orthonormal, sign-canonical
        assert np.abs(Vg.T @ Vg - np.eye(r)).max() < 1e-5
        idx = np.argmax(np.abs(basis[g]), axis=0)
        assert (basis[g][idx, np.arange(128)] > 0).all()
    if w.rank_k == 0:
        margins = []
        for g in range(w.n_groups):
            s = np.sqrt(f.lam[g])
            cum = np.cumsum(s) / s.sum()
            margins.append(abs(cum[f.group_ranks[g] - 1] - 0.9))
        if min(margins) > 1e-6:
            assert gr == f.group_ranks and rank == f.rank


def test_fit_energy_rank_modes(P):
    """Explicit spectra: the GPU picks the oracle's rank under both readings."""
    rng = np.random.default_rng(5)
    S, D = 4096, 128
    sigma = 10.0 / np.arange(1, D + 1)
    G = rng.standard_normal((S, D))
    U, _ = np.linalg.qr(G - G.mean(0))
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    x = (U @ np.diag(sigma) @ Q.T * 8 + 0.2).astype(np.float16).reshape(1, 1, S, D)
    for mode in (P.PALU_ENERGY_SIGMA, P.PALU_ENERGY_SIGMA2):
        cfg = P.palu_config_default(n_head_groups=1, rank=0, energy_mode=mode, energy_threshold=0.8)
        _, _, eig, rank, _ = P.fit(cfg, torch.from_numpy(x).to(DEV))
        f = O.fit(x.astype(np.float64), 1, rank=0, energy_threshold=0.8, energy_mode=mode)
        assert rank == f.rank


# ---------------------------------------------------------------- comparator

@pytest.mark.parametrize("S,Gq", [(1, 1), (63, 3), (1000, 7), (4097, 8)])
def test_fp16_comparator_matches_sdpa(P, S, Gq):
    rng = np.random.default_rng(S)
    B, H, cap = 2, 2, S + 30
    k = torch.from_numpy(rng.standard_normal((B, H, cap, 128)).astype(np.float16)).to(DEV)
    v = torch.from_numpy(rng.standard_normal((B, H, cap, 128)).astype(np.float16)).to(DEV)
    q = torch.from_numpy(rng.standard_normal((B, H * Gq, 128)).astype(np.float16)).to(DEV)
    ws = torch.empty(P.palu_fp16_decode_workspace_size(B, H, cap, H * Gq), dtype=torch.uint8, device=DEV)
    out = torch.empty(B, H * Gq, 128, dtype=torch.float32, device=DEV)
    P.palu_fp16_decode_attn(k, v, S, q, out, ws)
    kk = k[:, :, :S].double().repeat_interleave(Gq, dim=1)
    vv = v[:, :, :S].double().repeat_interleave(Gq, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double().unsqueeze(2), kk, vv).squeeze(2)
    err = O.relative_error(out.cpu().numpy(), ref.cpu().numpy())
    assert err.max() <= ATTN_TOL


# ---------------------------------------------------------------- errors and accounting

def test_capacity_and_length_errors(P):
    rng = np.random.default_rng(1)
    xk = rand_lowrank(rng, 1, 2, 40)
    cfg = P.palu_config_default(n_head_groups=1, rank=8)
    kc, vc = make_caches(P, cfg, cfg, xk, xk, 48)
    with pytest.raises(P.PaluError) as e:
        kc.append(torch.from_numpy(rand_lowrank(rng, 1, 2, 9)).to(DEV))
    assert e.value.status == 3
    kc.append(torch.from_numpy(rand_lowrank(rng, 1, 2, 1)).to(DEV))
    q = torch.zeros(1, 2, 128, dtype=torch.float16, device=DEV)
    with pytest.raises(P.PaluError):
        P.decode(kc, vc, q)
    assert kc.sync() == 0


def test_stats_against_oracle_accounting(P):
    rng = np.random.default_rng(2)
    x = rand_lowrank(rng, 2, 4, 100)
    cfg = P.palu_config_default(n_head_groups=2, rank=20)
    kc, _ = make_caches(P, cfg, cfg, x, x, 128)
    st = kc.stats()
    o = oracle_view(kc, O.ROLE_KEY).stats()
    assert st["code_bytes"] == o["code_bytes"] and st["meta_bytes"] == o["meta_bytes"]
    assert st["tail_bytes"] == o["tail_bytes"] and st["fp16_bytes"] == o["fp16_bytes"]
    assert st["effective_bits"] == pytest.approx(o["effective_bits"])
    assert st["code_bytes"] + st["meta_bytes"] + st["tail_bytes"] < st["fp16_bytes"]


def test_determinism(P):
    outs = []
    for _ in range(2):
        rng = np.random.default_rng(9)
        x = rand_lowrank(rng, 1, 4, 300, n_groups=2)
        cfg = P.palu_config_default(n_head_groups=2, rank=24)
        kc, vc = make_caches(P, cfg, cfg, x, x, 320)
        q = torch.from_numpy(rng.standard_normal((1, 12, 128)).astype(np.float16)).to(DEV)
        outs.append((kc.record_array()[:, :, :300 // 32], P.decode(kc, vc, q).cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
