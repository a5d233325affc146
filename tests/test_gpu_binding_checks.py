"""The Python binding refuses, before any launch, device tensors whose
pointer would not describe the buffer a C call reads or writes (the library
sees pointers and sizes only): another batch or head count than the cache's,
another dtype, a strided view, a token count that differs from the tensor's.
After the refusals every cache is as it was and decodes as before.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _h(rng, *shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float16)).to(DEV)


def test_latent_cache_calls_refuse_mismatched_tensors(P):
    rng = np.random.default_rng(31)
    B, H, S, r = 2, 4, 70, 24
    cfg = P.palu_config_default(n_head_groups=2, rank=r)
    x = _h(rng, B, H, S, 128)
    basis, mu, _, _, _ = P.fit(cfg, x)
    kc = P.LatentCache(cfg, P.PALU_ROLE_KEY, r, B, H, 128, basis, mu)
    vc = P.LatentCache(cfg, P.PALU_ROLE_VALUE, r, B, H, 128, basis, mu)
    kc.append(x)
    vc.append(x)
    q = _h(rng, B, 2 * H, 128)
    before = P.decode(kc, vc, q)
    rec_k, rec_v = kc.record_array().copy(), vc.record_array().copy()
    ws = torch.empty(P.palu_decode_workspace_size(kc.c, vc.c, 2 * H), dtype=torch.uint8, device=DEV)
    out = torch.empty(B, 2 * H, 128, dtype=torch.float32, device=DEV)
    one = _h(rng, B, H, 1, 128)
    refusals = [
        lambda: kc.append(_h(rng, B + 1, H, 3, 128)),                     # another batch
        lambda: kc.append(_h(rng, B, H - 1, 3, 128)),                     # another head count
        lambda: kc.append(_h(rng, B, H, 3, 128).float()),                 # fp32
        lambda: kc.append(_h(rng, B, 3, H, 128).transpose(1, 2)),         # strided view
        lambda: P.palu_encode_append(kc.c, _h(rng, B, H, 3, 128), 5),     # 5 tokens of a 3-token tensor
        lambda: P.palu_decode_attn(kc.c, vc.c, _h(rng, B + 1, 2 * H, 128), out, ws),
        lambda: P.palu_decode_attn(kc.c, vc.c, q.float(), out, ws),
        lambda: P.palu_decode_attn(kc.c, vc.c, q, out[:, :H], ws),        # out smaller than q
        lambda: P.palu_decode_attn(kc.c, vc.c, q, out.to(torch.bfloat16), ws),
        lambda: P.palu_decode_attn(kc.c, vc.c, q, out, torch.empty(ws.numel(), dtype=torch.int32, device=DEV)),
        lambda: P.palu_decode_attn_noalloc(kc.c, vc.c, q[:, ::2], out[:, :H]),
        lambda: P.palu_decode_step(kc.c, vc.c, _h(rng, B, H + 1, 128), one, q, out, ws),
        lambda: P.palu_decode_step(kc.c, vc.c, one, one[:, :, :, :64], q, out, ws),
        lambda: kc.append_ragged(_h(rng, B, H, 3, 128), torch.ones(B, dtype=torch.int64, device=DEV)),
        lambda: kc.append_ragged(_h(rng, B, H, 3, 128), torch.ones(B + 1, dtype=torch.int32, device=DEV)),
        lambda: kc.truncate_ragged(torch.full((B,), 64, dtype=torch.int32, device=DEV)),
        lambda: kc.restore(torch.zeros(1024, dtype=torch.uint8, device=DEV)),  # an image on the device
    ]
    for call in refusals:
        with pytest.raises(ValueError):
            call()
    torch.cuda.synchronize()
    assert kc.sync() == 0 and vc.sync() == 0 and kc.length == vc.length == S
    assert np.array_equal(kc.record_array(), rec_k) and np.array_equal(vc.record_array(), rec_v)
    assert torch.equal(P.decode(kc, vc, q), before)


def test_fit_calls_refuse_mismatched_outputs(P):
    rng = np.random.default_rng(32)
    cfg = P.palu_config_default(n_head_groups=2, rank=8)
    x = _h(rng, 1, 4, 64, 128)
    ws = torch.empty(P.palu_fit_workspace_size(cfg, 1, 4, 64), dtype=torch.uint8, device=DEV)
    basis = torch.empty(2, 128, 128, device=DEV)
    mu = torch.empty(2, 128, device=DEV)
    eig = torch.empty(2, 128, dtype=torch.float64, device=DEV)
    for args in [(x, ws, basis[:1], mu, eig), (x, ws, basis, mu, eig.float()), (x[..., :64], ws, basis, mu, eig),
                 (x.transpose(2, 3), ws, basis, mu, eig)]:
        with pytest.raises(ValueError):
            P.palu_fit(cfg, *args)
    with pytest.raises(ValueError):
        P.palu_fit_batch([cfg, cfg], [x, x], ws, [basis], [mu, mu], [eig, eig])   # one basis for two tensors
    with pytest.raises(ValueError):
        P.LatentCache(cfg, P.PALU_ROLE_KEY, 8, 1, 4, 64, basis[:, :, :8], mu, basis_ld=128)  # strided basis


def test_comparator_calls_refuse_mismatched_tensors(P):
    rng = np.random.default_rng(33)
    B, H, S = 1, 2, 40
    kv = P.KiviCache(B, H, 64, DEV)
    k = _h(rng, B, H, S, 128)
    kv.append(k, k)
    q = _h(rng, B, 2 * H, 128)
    ref = kv.decode(q)
    for call in (lambda: kv.append(k, k[:, :, :S - 1].contiguous()),           # keys and values differ
                 lambda: kv.append(_h(rng, B, H + 1, 2, 128), _h(rng, B, H + 1, 2, 128)),
                 lambda: kv.decode(_h(rng, B + 1, 2 * H, 128))):
        with pytest.raises(ValueError):
            call()
    assert kv.length == S and torch.equal(kv.decode(q), ref)
    ws = torch.empty(P.palu_fp16_decode_workspace_size(B, H, 64, 2 * H), dtype=torch.uint8, device=DEV)
    kf = _h(rng, B, H, 64, 128)
    out = torch.empty(B, 2 * H, 128, dtype=torch.float32, device=DEV)
    for call in (lambda: P.palu_fp16_decode_attn(kf, kf[:, :, :32].contiguous(), S, q, out, ws),
                 lambda: P.palu_fp16_decode_attn(kf, kf, S, q[:, :, :64].contiguous(), out, ws)):
        with pytest.raises(ValueError):
            call()
