"""palu_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory while they decode (a plugin whose host application
owns every allocation, a serving loop that forbids allocation between steps,
a process whose device memory another pool has reserved).  The entry point
keeps its split-K partials in a fixed array inside the library instead of a
caller workspace.  This file is collected last on purpose, so a run that
stops at the first failure has already run every other test.

Checked through the C ABI: two calls in a row (different queries and one
appended token between them, so a stale scratch would show) agree within the
attention tolerance with the CPU oracle on the stored codes and with the
workspace entry point, and a cache set whose partials exceed the fixed
scratch is refused with a clear error."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import palu
    palu.lib()
    return palu


def _lowrank(rng, B, H, S):
    A = rng.standard_normal((24, 128)) / math.sqrt(24)
    return (rng.standard_normal((B, H, S, 24)) @ A + rng.standard_normal(128) * 0.7).astype(np.float16)


def _oracle_view(c, role):
    Vr, mu = c.basis_array()
    cc = c.c
    return O.OracleCache.from_buffers(role, Vr, mu, cc.rank, cc.batch, cc.kv_heads, cc.capacity, bool(cc.quantize),
                                      c.record_array(), c.tail_array(), cc.length)


def test_noalloc_matches_oracle_and_workspace_decode_on_two_calls(P):
    rng = np.random.default_rng(42)
    B, H, Gq, S = 2, 4, 3, 301
    caches = []
    xs = []
    for role, r in ((P.PALU_ROLE_KEY, 24), (P.PALU_ROLE_VALUE, 28)):
        x = _lowrank(rng, B, H, S + 1)
        xs.append(x)
        cfg = P.palu_config_default(n_head_groups=2, rank=r)
        xt = torch.from_numpy(x[:, :, :S].copy()).to(DEV)
        basis, mu, _, rank, _ = P.fit(cfg, xt)
        c = P.LatentCache(cfg, role, rank, B, H, S + 16, basis, mu)
        c.append(xt)
        caches.append(c)
    kc, vc = caches
    lib = P.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        if call == 1:  # one more token between the calls
            kc.append(torch.from_numpy(xs[0][:, :, S:S + 1].copy()).to(DEV))
            vc.append(torch.from_numpy(xs[1][:, :, S:S + 1].copy()).to(DEV))
        q = torch.from_numpy(rng.standard_normal((B, H * Gq, 128)).astype(np.float16)).to(DEV)
        ref = P.decode(kc, vc, q, out_dtype=torch.float32)          # workspace entry point
        out = torch.full((B, H * Gq, 128), float("nan"), dtype=torch.float32, device=DEV)
        st = lib.palu_decode_attn_noalloc(ctypes.byref(kc.c), ctypes.byref(vc.c), ctypes.c_void_p(q.data_ptr()),
                                          H * Gq, ctypes.c_float(0.0), ctypes.c_void_p(out.data_ptr()), 1, stream)
        assert st == P.PALU_OK, P.palu_last_error()
        torch.cuda.synchronize()
        assert kc.sync() == 0 and vc.sync() == 0
        got = out.cpu().numpy()
        # the oracle: naive fp64 attention over K and V rebuilt from the stored codes
        ora = O.attend(q.cpu().numpy(), _oracle_view(kc, O.ROLE_KEY), _oracle_view(vc, O.ROLE_VALUE))
        err = O.relative_error(got, ora)
        assert np.isfinite(err).all() and err.max() <= ATTN_TOL, f"call {call} vs oracle: {err.max():.3e}"
        err_ws = O.relative_error(got, ref.cpu().numpy())
        assert np.isfinite(err_ws).all() and err_ws.max() <= ATTN_TOL, f"call {call} vs workspace: {err_ws.max():.3e}"


def test_noalloc_refuses_partials_larger_than_its_scratch(P):
    B, H, r, cap = 256, 8, 128, 64
    cfg = P.palu_config_default(n_head_groups=1, rank=r)
    q_heads = 8 * H
    basis = torch.linalg.qr(torch.randn(128, 128, dtype=torch.float64))[0].float().contiguous().to(DEV).unsqueeze(0)
    mu = torch.zeros(1, 128, dtype=torch.float32, device=DEV)
    kc = P.LatentCache(cfg, P.PALU_ROLE_KEY, r, B, H, cap, basis, mu)
    vc = P.LatentCache(cfg, P.PALU_ROLE_VALUE, r, B, H, cap, basis, mu)
    assert P.palu_decode_workspace_size(kc.c, vc.c, q_heads) > (4 << 20)
    q = torch.zeros(B, q_heads, 128, dtype=torch.float16, device=DEV)
    out = torch.empty(B, q_heads, 128, dtype=torch.float16, device=DEV)
    with pytest.raises(P.PaluError) as e:
        P.palu_decode_attn_noalloc(kc.c, vc.c, q, out)
    assert e.value.status == 2 and "scratch" in str(e.value)
