"""Pins for the CPU oracle: each checks the oracle against something other
than itself (closed forms from the pages, constructed inputs with known
answers, independent library routines, hand-worked cases, invariants)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.conftest import golden_path


# ---------------------------------------------------------------- closed forms

def test_effective_bits_closed_form():
    """PALU page, "Effective bit-width": (r/D)(0.25*4 + 0.75*2); 0.625 at r=32, D=128."""
    rows = [l.split() for l in open(golden_path("effective_bits.txt")) if l.strip() and not l.startswith("#")]
    assert rows
    for r, D, n_hi, bits in rows:
        r, D, n_hi, bits = int(r), int(D), int(n_hi), float(bits)
        assert O.n_hi_channels(r, 0.25) == n_hi
        assert O.effective_bits(r, D, n_hi) == pytest.approx(bits, abs=0)


def test_n_hi_is_top_quarter():
    # "top-25% latent channels (by singular value)" -> ceil(0.25 r)
    assert [O.n_hi_channels(r) for r in (1, 2, 3, 4, 5, 8, 27, 30, 52, 74, 128)] == \
           [1, 1, 1, 1, 2, 2, 7, 8, 13, 19, 32]
    assert O.n_hi_channels(10, 0.3) == 3          # 0.3*10 is 3.0000000000000004 in fp64
    assert O.n_hi_channels(7, 0.0) == 0 and O.n_hi_channels(7, 1.0) == 7


def test_assigned_avg_bits_below_two_at_default():
    """PALU page, "Evidence": assigned_avg_bits < 2.0 at default settings
    (r ~ 0.25 D through the threshold; K and V quantized)."""
    D = 128
    r = 32
    rate = O.effective_bits(r, D, O.n_hi_channels(r))
    assert max(rate, rate) < 2.0
    # values kept as fp16 latents: 16 r / D ("Effective bit-width")
    assert 16 * r / D == 4.0


# ---------------------------------------------------------------- quantizer

def _read_quant_cases():
    cases = []
    for line in open(golden_path("quantizer_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        bits, vals, sz, codes = [p.split() for p in line.split("|")]
        cases.append((int(bits[0]), np.array(vals, np.float64), float(sz[0]), float(sz[1]),
                      np.array(codes, np.int64)))
    return cases


@pytest.mark.parametrize("case", range(7))
def test_quantizer_hand_cases(case):
    bits, vals, s, z, codes = _read_quant_cases()[case]
    assert np.all(vals.astype(np.float32) == vals)          # inputs exact in fp32
    # put the group in channel 0; n_hi selects its bit width
    L = vals.astype(np.float32).reshape(1, 32, 1)
    n_hi = 1 if bits == 4 else 0
    q, s_h, z_h = O.quantize_blocks(L, n_hi, 4, 2)
    assert float(s_h[0, 0]) == s and float(z_h[0, 0]) == z
    assert np.array_equal(q[0, :, 0].astype(np.int64), codes)


def test_quantizer_range_and_error_bound():
    rng = np.random.default_rng(1)
    L = (rng.standard_normal((50, 32, 12)) * rng.uniform(0.01, 30, (50, 1, 12))).astype(np.float32)
    n_hi = 3
    q, s, z = O.quantize_blocks(L, n_hi)
    qmax = np.where(np.arange(12) < n_hi, 15, 3)
    assert (q <= qmax).all()
    deq = O.dequantize(q, s, z)
    # reconstruction error within half a step plus the fp16 rounding of scale/zero
    step = s.astype(np.float64)[:, None, :]
    err = np.abs(deq - L)
    bound = 0.5 * step + np.abs(z.astype(np.float64) - L.min(1))[:, None, :] + \
        qmax * np.abs(step - ((L.max(1) - L.min(1)) / qmax)[:, None, :]) + 1e-6
    assert (err <= bound).all()
    # min and max of every group are reproduced to within one step
    assert (np.abs(deq.min(1) - L.min(1)) <= s + 1e-6).all()


# ---------------------------------------------------------------- packing

def test_packing_is_lsb_first_with_2bit_shifts_0_2_4_6():
    """Blog "How I built VeloxQuant-MLX", "The Bit-Packing Problem": sub-byte
    codes go LSB-first; four 2-bit codes occupy shifts 0, 2, 4, 6 of a byte."""
    lay = O.Layout(O.ROLE_KEY, 32, 8)
    # channel 8 is the first 2-bit channel; tokens 0, 8, 16, 24 of lane 0 fill one byte
    assert [lay.code_position(t, 8) for t in (0, 8, 16, 24)] == \
           [(128, 0, 2), (128, 2, 2), (128, 4, 2), (128, 6, 2)]
    # 4-bit codes: two per byte, low nibble first
    assert [lay.code_position(t, 0) for t in (0, 8)] == [(0, 0, 4), (0, 4, 4)]


def test_packing_hand_positions():
    """Positions worked out by hand from the layout definition (key and value)."""
    k = O.Layout(O.ROLE_KEY, 32, 8)
    assert k.record_bytes == 128 * 1 + 64 * 3 + 4 * 32
    assert k.code_position(16, 1) == (3, 0, 4)      # field k=2, slot 1 -> high half, bit 24
    assert k.code_position(1, 2) == (20, 0, 4)      # token 1 -> g=1, slot 2 -> c=1: lane 5
    assert k.code_position(0, 16) == (130, 0, 2)    # second lo octet: upper halfword of the pair
    assert k.code_position(0, 9) == (129, 0, 2)     # slot 1 -> high byte of the halfword
    assert k.code_position(0, 24) == (256, 0, 2)    # third lo octet of three: the odd one, u16 per lane
    assert k.scale_zero_offsets(0) == (320, 320 + 64)
    v = O.Layout(O.ROLE_VALUE, 32, 8)
    assert v.code_position(1, 0) == (2, 0, 4)       # value: token parity -> high half (bit 16)
    assert v.code_position(2, 0) == (4, 0, 4)       # token 2 -> c=1: lane 1
    assert v.code_position(0, 3) == (48, 0, 4)      # slot 3 -> g=3: lane 12, byte 4*12
    assert v.code_position(8, 0) == (0, 4, 4)       # token 8 -> field 1
    assert v.scale_zero_offsets(1) == (324, 326)
    f = O.Layout(O.ROLE_VALUE, 32, 0, quantize=False)
    assert f.record_bytes == 4 * 512
    assert f.latent_offset(1, 9) == 512 + 16 * 4 + 2


@pytest.mark.parametrize("role", [O.ROLE_KEY, O.ROLE_VALUE])
@pytest.mark.parametrize("r", [1, 7, 8, 9, 16, 17, 27, 30, 32, 52, 74, 100, 128])
def test_pack_roundtrip_and_unique_positions(role, r):
    n_hi = O.n_hi_channels(r)
    lay = O.Layout(role, r, n_hi)
    rng = np.random.default_rng(r + 100 * role)
    maxc = np.where(np.arange(r) < n_hi, 16, 4)
    codes = (rng.integers(0, 1 << 16, (3, 32, r)) % maxc).astype(np.uint8)
    s = rng.standard_normal((3, r)).astype(np.float16)
    z = rng.standard_normal((3, r)).astype(np.float16)
    rec = lay.pack(codes, s, z)
    assert rec.shape == (3, lay.record_bytes) and lay.record_bytes % 16 == 0
    c2, s2, z2 = lay.unpack(rec)
    assert np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint16), s.view(np.uint16))
    assert np.array_equal(z2.view(np.uint16), z.view(np.uint16))
    seen = set()
    for t in range(32):
        for j in range(r):
            byte, sh, w = lay.code_position(t, j)
            assert byte < lay.sz_base and sh + w <= 8
            for b in range(w):
                assert (byte, sh + b) not in seen
                seen.add((byte, sh + b))
    # every pattern of one field round-trips on its own (exhaustive per width)
    for j in (0, r - 1):
        for val in range(int(maxc[j])):
            cc = np.zeros((1, 32, r), np.uint8)
            cc[0, 5, j] = val
            assert lay.unpack(lay.pack(cc, s[:1], z[:1]))[0][0, 5, j] == val
    f = O.Layout(role, r, 0, quantize=False)
    lat = rng.standard_normal((2, 32, r)).astype(np.float16)
    assert np.array_equal(f.unpack_latents(f.pack_latents(lat)).view(np.uint16), lat.view(np.uint16))


# ---------------------------------------------------------------- fit

def _constructed(n, sigma, rng, mu_scale=0.7):
    """X = U diag(sigma) Q^T + mu with U orthonormal, zero-mean columns: the
    centred Gram has eigenvalues sigma^2 and eigenvectors Q exactly."""
    D = len(sigma)
    G = rng.standard_normal((n, D))
    G -= G.mean(axis=0)
    U, _ = np.linalg.qr(G)
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    mu = rng.standard_normal(D) * mu_scale
    return U @ np.diag(sigma) @ Q.T + mu, Q, mu


@pytest.mark.parametrize("D", [4, 8, 64, 128])
def test_fit_recovers_constructed_spectrum(D):
    rng = np.random.default_rng(D)
    sigma = np.sort(rng.uniform(0.5, 10.0, D))[::-1] * np.linspace(1.0, 0.5, D)
    X, Q, mu = _constructed(4 * D + 16, sigma, rng)
    m, lam, V = O.fit_group(X)
    assert np.allclose(m, mu, atol=1e-12)
    assert np.allclose(lam, sigma ** 2, rtol=1e-9)
    assert np.allclose(np.abs(V.T @ Q), np.eye(D), atol=1e-8)
    # canonical sign: the largest-|.| entry of each direction is positive
    idx = np.argmax(np.abs(V), axis=0)
    assert (V[idx, np.arange(D)] > 0).all()


@pytest.mark.parametrize("S,D", [(64, 4), (64, 8), (40, 128), (300, 128)])
def test_fit_matches_svd_of_centred_rows(S, D):
    """SVD-versus-eigendecomposition equivalence: the right singular vectors and
    squared singular values of X_c (numpy SVD) equal the oracle's fit."""
    rng = np.random.default_rng(S * D)
    X = rng.standard_normal((S, D)) @ np.diag(np.linspace(3, 0.1, D)) + rng.standard_normal(D)
    mu, lam, V = O.fit_group(X)
    _, sv, Vt = np.linalg.svd(X - X.mean(0), full_matrices=False)
    k = min(S - 1, D)          # directions with nonzero singular values
    assert np.allclose(lam[:k], sv[:k] ** 2, rtol=1e-8)
    assert np.allclose(lam[k:], 0.0, atol=1e-8 * lam[0])
    assert np.allclose(np.abs(np.sum(V[:, :k] * Vt[:k].T, axis=0)), 1.0, atol=1e-7)


def test_energy_rank_brute_force():
    """Ranks from hand cumulative sums. sigma = (4, 3, 2, 1):
    sigma reading: 0.4, 0.7, 0.9, 1.0;  sigma^2 reading: 16/30, 25/30, 29/30, 1."""
    lam = np.array([16.0, 9.0, 4.0, 1.0])
    S, S2 = O.ENERGY_SIGMA, O.ENERGY_SIGMA2
    assert [O.energy_rank(lam, t, S) for t in (0.3, 0.65, 0.85, 0.95)] == [1, 2, 3, 4]
    assert [O.energy_rank(lam, t, S2) for t in (0.5, 0.8, 0.85, 0.99)] == [1, 2, 3, 4]
    assert O.energy_rank(np.zeros(8), 0.9) == 1
    assert O.energy_rank(lam, 1.0, S) == 4


def test_energy_rank_on_constructed_data_both_readings():
    rng = np.random.default_rng(7)
    D = 32
    sigma = 1.0 / np.arange(1, D + 1)
    X, _, _ = _constructed(256, sigma, rng)
    _, lam, _ = O.fit_group(X)
    c1 = np.cumsum(sigma) / sigma.sum()
    c2 = np.cumsum(sigma ** 2) / (sigma ** 2).sum()
    for tau in (0.5, 0.8, 0.9):
        # thresholds away from the cumulative values so rounding cannot decide
        assert np.min(np.abs(c1 - tau)) > 1e-6 and np.min(np.abs(c2 - tau)) > 1e-6
        assert O.energy_rank(lam, tau, O.ENERGY_SIGMA) == int(np.argmax(c1 >= tau)) + 1
        assert O.energy_rank(lam, tau, O.ENERGY_SIGMA2) == int(np.argmax(c2 >= tau)) + 1
    # "Energy-threshold rank selection returns a rank in [1, D]"
    for _ in range(20):
        lam = np.sort(rng.exponential(1.0, D))[::-1]
        assert 1 <= O.energy_rank(lam, rng.uniform(0, 1), O.ENERGY_SIGMA) <= D


def test_fit_groups_and_min_rank():
    """Contiguous head groups; one rank = min over groups; explicit rank wins."""
    rng = np.random.default_rng(3)
    B, H, S, D = 2, 4, 40, 16
    x = np.zeros((B, H, S, D))
    true_rank = [3, 6]                                  # group 0 heads 0-1, group 1 heads 2-3
    for g, tr in enumerate(true_rank):
        A = rng.standard_normal((tr, D))
        z = rng.standard_normal((B, 2, S, tr))
        z -= z.reshape(-1, tr).mean(axis=0)          # zero mean over the group's stacked rows
        x[:, 2 * g:2 * g + 2] = z @ A + (0.5 + g)
    f = O.fit(x, 2, rank=0, energy_threshold=0.999999, energy_mode=O.ENERGY_SIGMA2)
    assert f.group_ranks == true_rank and f.rank == 3
    assert np.allclose(f.mu[0], 0.5, atol=1e-12) and np.allclose(f.mu[1], 1.5, atol=1e-12)
    assert O.fit(x, 2, rank=5).rank == 5 and O.fit(x, 2, rank=500).rank == D


def test_planted_subspace_recovery_mse():
    """PALU page, "Evidence": group SVD recovers a planted rank-r subspace to MSE < 1e-3."""
    rng = np.random.default_rng(11)
    D, r = 64, 8
    A = rng.standard_normal((r, D))
    X = rng.standard_normal((2048, r)) @ A + rng.standard_normal(D)
    noisy = X + 1e-3 * rng.standard_normal(X.shape)
    mu, lam, V = O.fit_group(noisy)
    Vr = V[:, :r]
    rec = (noisy - mu) @ Vr @ Vr.T + mu
    assert np.mean((rec - X) ** 2) < 1e-3
    # and the planted row space is recovered
    Qa, _ = np.linalg.qr(A.T)
    assert O.subspace_residual(Qa, Vr) < 1e-3


def _naive_2bit_mse(x):
    """Per-channel 2-bit min/max quantization of the raw [S, D] data in 32-token groups."""
    S, D = x.shape
    blocks = x.reshape(S // 32, 32, D).astype(np.float32)
    q, s, z = O.quantize_blocks(blocks, 0, 4, 2)
    return float(np.mean((O.dequantize(q, s, z).reshape(S, D) - x) ** 2))


def test_planted_rank8_beats_naive_2bit():
    """PALU page, "Evidence": on rank-8 data (D=64), rank 8 latents (mixed 4/2-bit)
    have lower reconstruction MSE than naive 2-bit, for keys and for values."""
    rng = np.random.default_rng(5)
    D, r, S = 64, 8, 1024
    for tensor in range(2):
        A = rng.standard_normal((r, D)) / math.sqrt(r)
        x = (rng.standard_normal((1, 1, S, r)) @ A + rng.standard_normal(D) * 0.5).astype(np.float16)
        f = O.fit(x.astype(np.float64), 1, rank=r)
        c = O.OracleCache(tensor, f.basis.astype(np.float32), f.mu.astype(np.float32), r, 1, 1, S)
        c.append(x)
        rec = c.reconstruct(0, 0)
        mse_palu = float(np.mean((rec - x[0, 0]) ** 2))
        assert mse_palu < _naive_2bit_mse(x[0, 0].astype(np.float64))


# ---------------------------------------------------------------- reconstruction / attention

def test_full_rank_unquantized_reconstruction_is_exact():
    """r = D with fp64 latents: (x - mu) V V^T + mu = x."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((300, 32)) * 3 + 1
    mu, lam, V = O.fit_group(x)
    rec = (x - mu) @ V @ V.T + mu
    assert np.max(np.abs(rec - x)) < 1e-12


def _small_caches(quantize_v=True, S=77, r=12, Hkv=4, n_groups=2, B=2, seed=0):
    rng = np.random.default_rng(seed)
    D = 32
    xk = (rng.standard_normal((B, Hkv, S, 8)) @ rng.standard_normal((8, D)) + 0.3).astype(np.float16)
    xv = (rng.standard_normal((B, Hkv, S, 8)) @ rng.standard_normal((8, D)) - 0.2).astype(np.float16)
    fk = O.fit(xk, n_groups, rank=r)
    fv = O.fit(xv, n_groups, rank=r)
    kc = O.OracleCache(O.ROLE_KEY, fk.basis.astype(np.float32), fk.mu.astype(np.float32), r, B, Hkv, 128)
    vc = O.OracleCache(O.ROLE_VALUE, fv.basis.astype(np.float32), fv.mu.astype(np.float32), r, B, Hkv, 128,
                       quantize=quantize_v)
    kc.append(xk)
    vc.append(xv)
    return kc, vc, rng


@pytest.mark.parametrize("quantize_v", [True, False])
def test_latent_attention_equals_reconstructed_attention(quantize_v):
    """softmax(q K_hat^T) V_hat equals the latent-space evaluation (q~ = q V_g,
    c = q.mu_g, weighted sum of L_hat then V_g^T + mu_g), since sum(p) = 1."""
    kc, vc, rng = _small_caches(quantize_v)
    q = rng.standard_normal((2, 12, 32)).astype(np.float16)
    a = O.attend(q, kc, vc)
    b = O.attend_latent(q, kc, vc)
    assert np.max(np.abs(a - b)) < 1e-11


def test_attention_matches_torch_sdpa():
    """Naive fp64 attention over the reconstructed cache vs torch's SDPA (fp64, CPU)."""
    kc, vc, rng = _small_caches(True)
    q = rng.standard_normal((2, 8, 32)).astype(np.float16)   # GQA 2:1
    out = O.attend(q, kc, vc)
    for b in range(2):
        for h in range(8):
            K = torch.from_numpy(kc.reconstruct(b, h // 2))
            V = torch.from_numpy(vc.reconstruct(b, h // 2))
            qq = torch.from_numpy(q[b, h].astype(np.float64)).view(1, 1, 1, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(qq, K[None, None], V[None, None])
            assert np.allclose(out[b, h], ref.view(-1).numpy(), rtol=1e-12, atol=1e-12)


def test_gqa_mapping_uses_each_query_heads_own_kv_head():
    """Query head h reads KV head h // Gq for every h (not only the first of a group)."""
    kc, vc, rng = _small_caches(True, Hkv=4)
    q = rng.standard_normal((2, 12, 32)).astype(np.float16)  # Gq = 3
    out = O.attend(q, kc, vc)
    for h in range(12):
        single = O.attend(q[:, h:h + 1].repeat(3, axis=1)[:, :1].repeat(1, axis=1), _one_head(kc, h // 3),
                          _one_head(vc, h // 3))
        assert np.allclose(out[:, h], single[:, 0], rtol=1e-13, atol=1e-13)


def _one_head(c, h):
    """A one-KV-head view of cache c holding stream h."""
    d = O.OracleCache.__new__(O.OracleCache)
    d.__dict__.update(c.__dict__)
    d.Hkv = 1
    d.blocks = c.blocks[:, h:h + 1]
    d.tail = c.tail[:, h:h + 1]
    g = c.group_of(h)
    d.V = c.V[g:g + 1]
    d.mu = c.mu[g:g + 1]
    d.n_groups = 1
    return d


# ---------------------------------------------------------------- cache invariants

@pytest.mark.parametrize("quantize", [True, False])
def test_prefill_then_appends_equals_one_prefill(quantize):
    rng = np.random.default_rng(9)
    B, H, D, r = 1, 2, 32, 10
    x = (rng.standard_normal((B, H, 100, D))).astype(np.float16)
    f = O.fit(x[:, :, :60].astype(np.float64), 1, rank=r)
    args = (O.ROLE_VALUE, f.basis.astype(np.float32), f.mu.astype(np.float32), r, B, H, 128)
    a = O.OracleCache(*args, quantize=quantize)
    a.append(x[:, :, :45])
    for t in range(45, 100):
        a.append(x[:, :, t:t + 1])
    b = O.OracleCache(*args, quantize=quantize)
    b.append(x)
    assert a.length == b.length == 100
    assert np.array_equal(a.blocks, b.blocks)
    assert np.array_equal(a.tail[:, :, :100 % 32], b.tail[:, :, :100 % 32])


def test_decode_offset_and_no_nans():
    """PALU "Evidence": decode produces valid output, offset grows by the steps."""
    kc, vc, rng = _small_caches(True, S=40)
    for step in range(30):
        kc.append(rng.standard_normal((2, 4, 1, 32)).astype(np.float16))
        vc.append(rng.standard_normal((2, 4, 1, 32)).astype(np.float16))
        out = O.attend(rng.standard_normal((2, 4, 32)).astype(np.float16), kc, vc)
        assert np.isfinite(out).all()
    assert kc.length == vc.length == 70


def test_byte_accounting_compressed_below_fp16():
    """PALU "Evidence": compressed key and value bytes < fp16 bytes, also with
    values kept as fp16 latents."""
    for qv in (True, False):
        kc, vc, _ = _small_caches(qv)
        for c in (kc, vc):
            st = c.stats()
            assert st["code_bytes"] + st["meta_bytes"] + st["tail_bytes"] < st["fp16_bytes"]


def test_determinism():
    """PALU "Evidence": two caches on the same data give identical output."""
    a = _small_caches(True, seed=4)
    b = _small_caches(True, seed=4)
    assert np.array_equal(a[0].blocks, b[0].blocks) and np.array_equal(a[1].blocks, b[1].blocks)
    q = np.random.default_rng(0).standard_normal((2, 4, 32)).astype(np.float16)
    assert np.array_equal(O.attend(q, a[0], a[1]), O.attend(q, b[0], b[1]))


def test_latent_storage_shape():
    """PALU "Evidence": buffers hold [S, r] latents, never the [S, D] tensor."""
    kc, vc, _ = _small_caches(True, S=64, r=12)
    assert kc.latents(0, 0).shape == (64, 12)
    assert kc.blocks.shape[-1] < 32 * 32 * 2         # a block record is far below 32 fp16 rows


def test_projection_inverts_on_a_full_basis():
    """L = (x - mu) V rounded to fp32; with the full orthonormal basis,
    L V^T + mu gives x back to within the fp32 rounding of L."""
    rng = np.random.default_rng(12)
    D = 64
    x = (rng.standard_normal((50, D)) * 2 + 0.3).astype(np.float16)
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    V = Q.astype(np.float32)
    mu = rng.standard_normal(D).astype(np.float32)
    L = O.project(x, V, mu)
    assert L.dtype == np.float32
    exact = (x.astype(np.float64) - mu.astype(np.float64)) @ V.astype(np.float64)
    assert np.all(np.abs(L - exact) <= np.abs(exact) * 2.0 ** -24 + 1e-30)
    back = L.astype(np.float64) @ V.astype(np.float64).T + mu
    assert np.max(np.abs(back - x.astype(np.float64))) < 1e-5


# ------------------------------------------------------------ small helpers

def test_canonical_sign_hand_cases():
    """Each column's largest-|.| entry ends positive; among equal magnitudes
    the lowest row index decides; a zero column is left as it is."""
    V = np.array([[0.6, -0.5, 0.0],
                  [-0.8, 0.5, 0.0],
                  [0.0, -0.7071, 0.0]])
    W = O.canonical_sign(V)
    assert np.array_equal(W[:, 0], [-0.6, 0.8, 0.0])
    assert np.array_equal(W[:, 1], [0.5, -0.5, 0.7071])
    assert np.array_equal(W[:, 2], [0.0, 0.0, 0.0])
    tie = np.array([[-0.5], [0.5], [0.1]])           # |-0.5| == |0.5|: row 0 decides
    assert np.array_equal(O.canonical_sign(tie)[:, 0], [0.5, -0.5, -0.1])


def test_subspace_residual_closed_form():
    """Two lines in the plane at angle t: the residual is |sin t|; a set
    against itself (any basis of it) is 0; orthogonal sets give sqrt(k)."""
    for t in (0.0, 0.3, 1.0, math.pi / 2):
        a = np.array([[1.0], [0.0]])
        b = np.array([[math.cos(t)], [math.sin(t)]])
        assert abs(O.subspace_residual(a, b) - abs(math.sin(t))) < 1e-14
    rng = np.random.default_rng(2)
    Q, _ = np.linalg.qr(rng.standard_normal((10, 10)))
    R, _ = np.linalg.qr(rng.standard_normal((3, 3)))
    assert O.subspace_residual(Q[:, :3], Q[:, :3] @ R) < 1e-13
    assert abs(O.subspace_residual(Q[:, :3], Q[:, 3:7]) - 2.0) < 1e-13


def test_relative_error_hand_case():
    ref = np.array([[[3.0, 4.0]], [[0.0, 2.0]]])     # norms 5 and 2
    out = np.array([[[3.5, 4.0]], [[0.0, 1.0]]])
    assert np.allclose(O.relative_error(out, ref), [[0.1], [0.5]], rtol=0, atol=1e-15)


def test_group_rows_brute_force():
    """Rows of group g are all (batch, head in g, token) vectors, batch-major."""
    B, H, S, D = 2, 6, 3, 4
    x = np.arange(B * H * S * D, dtype=np.float64).reshape(B, H, S, D)
    for n_groups in (1, 2, 3, 6):
        hg = H // n_groups
        for g in range(n_groups):
            want = [x[b, h, s] for b in range(B) for h in range(g * hg, (g + 1) * hg) for s in range(S)]
            assert np.array_equal(O.group_rows(x, n_groups, g), np.array(want))
