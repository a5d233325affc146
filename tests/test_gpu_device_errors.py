"""Device-side error reporting, exercised without faulting the GPU.

Conditions only the device can see set bits of a cache's device error word,
which palu_cache_sync reports (PALU_ERR_DEVICE) and clears:

- a bounded wait that runs out (PALU_DEVERR_TIMEOUT): the library's wait on
  a shared-memory barrier that nothing completes, with a short limit and no
  copy in flight, through the palu_debug_wait_probe hook;
- an append past capacity that the host could not refuse because it runs
  from a replayed CUDA graph (PALU_DEVERR_CAPACITY): nothing is written;
- key and value caches whose device lengths differ at decode
  (PALU_DEVERR_LENGTH_MISMATCH), made by replaying only the key append of a
  captured pair.

After each, the context stays usable: a later decode matches the oracle.
"""
import ctypes
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


def _raw_sync(P, cache):
    bits = ctypes.c_uint32()
    st = P.lib().palu_cache_sync(ctypes.byref(cache.c), ctypes.byref(bits),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, bits.value


def _caches(P, rng, B=1, H=2, S=40, cap=64, r=16):
    basis = torch.linalg.qr(torch.from_numpy(rng.standard_normal((128, 128))))[0].float().contiguous().to(DEV).unsqueeze(0)
    mu = torch.from_numpy(rng.standard_normal((1, 128)).astype(np.float32)).to(DEV)
    cfg = P.palu_config_default(n_head_groups=1, rank=r)
    kc = P.LatentCache(cfg, P.PALU_ROLE_KEY, r, B, H, cap, basis, mu)
    vc = P.LatentCache(cfg, P.PALU_ROLE_VALUE, r, B, H, cap, basis, mu)
    for c in (kc, vc):
        c.append(torch.from_numpy(rng.standard_normal((B, H, S, 128)).astype(np.float16)).to(DEV))
    return kc, vc


def _oracle_view(c, role):
    Vr, mu = c.basis_array()
    cc = c.c
    return O.OracleCache.from_buffers(role, Vr, mu, cc.rank, cc.batch, cc.kv_heads, cc.capacity, bool(cc.quantize),
                                      c.record_array(), c.tail_array(), cc.length)


def _decode_matches_oracle(P, kc, vc, rng, Gq=2):
    B, H = kc.c.batch, kc.c.kv_heads
    q = torch.from_numpy(rng.standard_normal((B, H * Gq, 128)).astype(np.float16)).to(DEV)
    out = P.decode(kc, vc, q, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kc.sync() == 0 and vc.sync() == 0
    ref = O.attend(q.cpu().numpy(), _oracle_view(kc, O.ROLE_KEY), _oracle_view(vc, O.ROLE_VALUE))
    err = O.relative_error(out.cpu().numpy(), ref)
    assert np.isfinite(err).all() and err.max() <= 2e-3


def test_bounded_wait_that_runs_out_sets_the_timeout_bit(P):
    rng = np.random.default_rng(7)
    kc, vc = _caches(P, rng)
    assert kc.sync() == 0
    P.palu_debug_wait_probe(kc.c, 2000, signal=False)       # nothing completes the barrier
    st, bits = _raw_sync(P, kc)
    assert st == 6 and bits == P.PALU_DEVERR_TIMEOUT, (st, bits)
    st, bits = _raw_sync(P, kc)                             # reported once, then cleared
    assert st == 0 and bits == 0
    P.palu_debug_wait_probe(kc.c, 2000, signal=True)        # completed barrier: no error
    st, bits = _raw_sync(P, kc)
    assert st == 0 and bits == 0
    _decode_matches_oracle(P, kc, vc, rng)


def test_replayed_append_past_capacity_sets_the_capacity_bit(P):
    rng = np.random.default_rng(8)
    cap = 60                                                 # the last block stays partial
    kc, vc = _caches(P, rng, S=cap - 1, cap=cap)
    one = torch.from_numpy(rng.standard_normal((1, 2, 1, 128)).astype(np.float16)).to(DEV)
    kc.append(one)                                           # warm the one-token path outside capture
    kc.truncate(cap - 1)
    assert kc.sync() == 0 and kc.c.length == cap - 1
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kc.append(one, stream=s)                             # the host count reaches the capacity
    g.replay()
    torch.cuda.synchronize()
    assert kc.sync() == 0 and kc.c.length == cap
    rec, tail = kc.record_array().copy(), kc.tail_array().copy()
    g.replay()                                               # one token past capacity, seen on the device only
    torch.cuda.synchronize()
    st, bits = _raw_sync(P, kc)
    assert st == 6 and bits == P.PALU_DEVERR_CAPACITY, (st, bits)
    assert kc.c.length == cap
    assert np.array_equal(kc.record_array(), rec) and np.array_equal(kc.tail_array(), tail)
    # the value cache is one token behind; bring it level and decode
    vc.append(one)
    _decode_matches_oracle(P, kc, vc, rng)


def test_kv_length_mismatch_at_decode_sets_its_bit(P):
    rng = np.random.default_rng(9)
    kc, vc = _caches(P, rng, S=45)
    one_k = torch.from_numpy(rng.standard_normal((1, 2, 1, 128)).astype(np.float16)).to(DEV)
    one_v = torch.from_numpy(rng.standard_normal((1, 2, 1, 128)).astype(np.float16)).to(DEV)
    kc.append(one_k)                                         # warm the one-token path outside capture
    vc.append(one_v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gk, gv = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=s):
        kc.append(one_k, stream=s)
    with torch.cuda.graph(gv, stream=s):
        vc.append(one_v, stream=s)
    assert kc.c.length == vc.c.length == 47                  # the host counts agree ...
    gk.replay()                                              # ... the device lengths will not
    torch.cuda.synchronize()
    q = torch.from_numpy(rng.standard_normal((1, 4, 128)).astype(np.float16)).to(DEV)
    P.decode(kc, vc, q, out_dtype=torch.float32)
    torch.cuda.synchronize()
    st, bits = _raw_sync(P, kc)
    assert st == 6 and bits == P.PALU_DEVERR_LENGTH_MISMATCH, (st, bits)
    gv.replay()                                              # level again
    torch.cuda.synchronize()
    assert vc.sync() == 0 and kc.c.length == vc.c.length == 47
    _decode_matches_oracle(P, kc, vc, rng)
