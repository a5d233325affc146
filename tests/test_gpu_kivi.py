"""KIVI-2bit comparator, GPU path vs the CPU oracle (oracle.kivi_oracle),
through the C ABI.

Bars: block records (codes, fp16 scale and zero) and window rows bit-exact;
decode attention within the same 2e-3 bar as the latent cache (max-abs error
relative to the output's L2 norm; the kernel rounds code * scale + zero to
fp16 once and the weights to fp16, the oracle is fp64 on the same codes).
"""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import kivi_oracle as K
from test_gpu_parity import ATTN_TOL, DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _kv(rng, B, H, S, scale=1.0):
    k = (scale * rng.standard_normal((B, H, S, 128)) + rng.standard_normal((1, 1, 1, 128))).astype(np.float16)
    v = (rng.standard_normal((B, H, S, 128)) * rng.uniform(0.2, 3.0, (B, H, S, 1))).astype(np.float16)
    return k, v


def _check_storage(c, oc):
    nb = oc.n_blocks
    assert c.length == oc.length
    got = c.record_array()[:, :, :nb]
    assert np.array_equal(got, K.records(oc)), "records differ"
    w = oc.length % 32
    win = c.window_array()
    assert np.array_equal(win[:, :, 0, :w], oc.window_k) and np.array_equal(win[:, :, 1, :w], oc.window_v)


@pytest.mark.parametrize("B,H,chunks", [(1, 1, (32,)), (2, 3, (77,)), (1, 2, (5, 27, 1, 40, 64, 3)),
                                        (3, 1, (1,) * 33), (2, 2, (300, 31, 1))])
def test_records_and_window_bit_exact(P, B, H, chunks):
    rng = np.random.default_rng(sum(chunks) + B)
    S = sum(chunks)
    k, v = _kv(rng, B, H, S)
    c = P.KiviCache(B, H, S + 5, DEV)
    oc = K.KiviCache(B, H)
    t = 0
    for n in chunks:
        c.append(torch.from_numpy(k[:, :, t:t + n].copy()).to(DEV), torch.from_numpy(v[:, :, t:t + n].copy()).to(DEV))
        oc.append(k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
    torch.cuda.synchronize()
    _check_storage(c, oc)


@pytest.mark.parametrize("S", [1, 5, 31, 32, 33, 64, 65, 100, 300, 1000, 2048 + 17])
@pytest.mark.parametrize("Gq", [1, 7])
def test_decode_matches_oracle(P, S, Gq):
    rng = np.random.default_rng(S * 10 + Gq)
    B, H = 2, 2
    k, v = _kv(rng, B, H, S)
    c = P.KiviCache(B, H, S, DEV)
    c.append(torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    oc = K.KiviCache(B, H)
    oc.append(k, v)
    q = rng.standard_normal((B, H * Gq, 128)).astype(np.float16)
    out = c.decode(torch.from_numpy(q).to(DEV))
    ref = K.kivi_attend(q, oc)
    err = O.relative_error(out.cpu().numpy(), ref)
    assert err.max() <= ATTN_TOL, f"max rel err {err.max():.3e}"


@pytest.mark.parametrize("Gq", [2, 4, 8])
def test_decode_gqa_factors_and_fp16_output(P, Gq):
    rng = np.random.default_rng(Gq)
    B, H, S = 1, 3, 700
    k, v = _kv(rng, B, H, S, scale=2.0)
    c = P.KiviCache(B, H, S + 100, DEV)
    c.append(torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    oc = K.KiviCache(B, H)
    oc.append(k, v)
    q = rng.standard_normal((B, H * Gq, 128)).astype(np.float16)
    out = c.decode(torch.from_numpy(q).to(DEV), out_dtype=torch.float16, softmax_scale=0.05)
    ref = K.kivi_attend(q, oc, scale=0.05)
    assert O.relative_error(out.float().cpu().numpy(), ref).max() <= ATTN_TOL


def test_decode_peaked_attention_and_determinism(P):
    """One key far more aligned with q than the rest: the output is that
    token's value; and repeated calls are bit-identical."""
    rng = np.random.default_rng(9)
    B, H, S = 2, 2, 500
    k, v = _kv(rng, B, H, S, scale=0.1)
    q = rng.standard_normal((B, H, 128)).astype(np.float16)
    for b in range(B):
        for h in range(H):
            k[b, h, 123] = (q[b, h].astype(np.float32) * 0.5).astype(np.float16)
    c = P.KiviCache(B, H, S, DEV)
    c.append(torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    oc = K.KiviCache(B, H)
    oc.append(k, v)
    qd = torch.from_numpy(q).to(DEV)
    out = c.decode(qd)
    ref = K.kivi_attend(q, oc)
    assert O.relative_error(out.cpu().numpy(), ref).max() <= ATTN_TOL
    assert all(torch.equal(out, c.decode(qd)) for _ in range(3))


def test_capacity_refused_and_length_kept(P):
    c = P.KiviCache(1, 1, 40, DEV)
    x = torch.zeros(1, 1, 40, 128, dtype=torch.float16, device=DEV)
    c.append(x, x)
    with pytest.raises(P.PaluError) as e:
        c.append(x[:, :, :1], x[:, :, :1])
    assert e.value.status == 3 and c.length == 40


def test_full_size_sampled_streams(P):
    """The benchmark's shape (batch 16, 4 KV heads, 7 query heads per KV head,
    32768 + 17 tokens, one layer): two sampled streams against the oracle,
    which sees only those streams' tokens."""
    from rank_latent_kv_gb300 import synth
    w = synth.WORKLOADS["qwen7b"]
    S = 32768 + 17
    g = torch.Generator(device=DEV).manual_seed(5)
    k = torch.randn(w.batch, w.hkv, S, 128, generator=g, device=DEV, dtype=torch.float32).half()
    v = (torch.randn(w.batch, w.hkv, S, 128, generator=g, device=DEV) * 2).half()
    c = P.KiviCache(w.batch, w.hkv, S, DEV)
    c.append(k, v)
    q = torch.randn(w.batch, w.hq, 128, generator=g, device=DEV).half()
    out = c.decode(q).cpu().numpy()
    Gq = w.hq // w.hkv
    for b, h in ((0, 0), (w.batch - 1, w.hkv - 1)):
        oc = K.KiviCache(1, 1)
        oc.append(k[b:b + 1, h:h + 1].cpu().numpy(), v[b:b + 1, h:h + 1].cpu().numpy())
        qs = q[b:b + 1, h * Gq:(h + 1) * Gq].cpu().numpy()
        ref = K.kivi_attend(qs, oc)
        err = O.relative_error(out[b:b + 1, h * Gq:(h + 1) * Gq], ref)
        assert err.max() <= ATTN_TOL, f"stream ({b},{h}): max rel err {err.max():.3e}"
        rec = c.record_array()[b, h, :oc.n_blocks]
        assert np.array_equal(rec, K.records(oc)[0, 0])
