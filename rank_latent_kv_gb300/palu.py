"""Thin ctypes binding of libpalu (include/palu.h, include/kivi.h).

Argument marshalling only: every step of the fit, append and decode runs in
the library's CUDA kernels.  PyTorch provides device memory and the current
stream.  If the library is missing the import of any entry point raises; there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_double, c_float, c_int32, c_int64, c_size_t, c_uint32, c_void_p, POINTER

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpalu.so")

PALU_OK = 0
PALU_ENERGY_SIGMA = 0
PALU_ENERGY_SIGMA2 = 1
PALU_ROLE_KEY = 0
PALU_ROLE_VALUE = 1
PALU_DEVERR_CAPACITY = 1
PALU_DEVERR_TIMEOUT = 2
PALU_DEVERR_LENGTH_MISMATCH = 4
PALU_DEVERR_NOT_CONVERGED = 8
PALU_DEVERR_ROLLBACK = 16
PALU_DEVERR_BOUNDS = 32
STATUS_NAMES = {0: "PALU_OK", 1: "PALU_ERR_INVALID_ARG", 2: "PALU_ERR_UNSUPPORTED", 3: "PALU_ERR_CAPACITY",
                4: "PALU_ERR_NOT_INITIALIZED", 5: "PALU_ERR_CUDA", 6: "PALU_ERR_DEVICE"}


class palu_config(ctypes.Structure):
    _fields_ = [("head_dim", c_int32), ("n_head_groups", c_int32), ("rank", c_int32), ("energy_mode", c_int32),
                ("energy_threshold", c_double), ("hi_fraction", c_double), ("hi_bit", c_int32),
                ("lo_bit", c_int32), ("group_size", c_int32), ("quantize", c_int32)]


class palu_cache(ctypes.Structure):
    _fields_ = [("magic", c_int32), ("role", c_int32), ("head_dim", c_int32), ("rank", c_int32),
                ("n_hi", c_int32), ("n_groups", c_int32), ("heads_per_group", c_int32), ("quantize", c_int32),
                ("batch", c_int32), ("kv_heads", c_int32), ("n_hi_oct", c_int32), ("n_lo_oct", c_int32),
                ("n_oct", c_int32), ("record_bytes", c_int32), ("capacity", c_int64), ("n_blk_cap", c_int64),
                ("blocks", c_void_p), ("tail", c_void_p), ("state", c_void_p), ("length", c_int64)]


class palu_stats(ctypes.Structure):
    _fields_ = [("length", c_int64), ("rank", c_int32), ("n_hi", c_int32), ("code_bytes", c_double),
                ("meta_bytes", c_double), ("tail_bytes", c_double), ("record_bytes", c_double),
                ("basis_bytes", c_double), ("fp16_bytes", c_double), ("effective_bits", c_double),
                ("bits_with_meta", c_double)]


class palu_kivi_cache(ctypes.Structure):
    _fields_ = [("magic", c_int32), ("batch", c_int32), ("kv_heads", c_int32), ("bits", c_int32),
                ("capacity", c_int64), ("n_blk_cap", c_int64), ("records", c_void_p), ("window", c_void_p),
                ("length", c_int64)]


class palu_svdq_cache(ctypes.Structure):
    _fields_ = [("magic", c_int32), ("batch", c_int32), ("kv_heads", c_int32), ("r_max", c_int32),
                ("record_bytes", c_int32), ("pad0", c_int32), ("capacity", c_int64), ("n_blk_cap", c_int64),
                ("blocks", c_void_p), ("tail", c_void_p), ("state", c_void_p), ("length", c_int64)]


_P = POINTER
_SIGNATURES = {
    "palu_last_error": (ctypes.c_char_p, []),
    "palu_version": (ctypes.c_char_p, []),
    "palu_config_default": (c_int32, [_P(palu_config)]),
    "palu_fit_workspace_size": (c_int32, [_P(palu_config), c_int64, c_int32, c_int64, _P(c_size_t)]),
    "palu_fit": (c_int32, [_P(palu_config), c_void_p, c_int64, c_int32, c_int64, c_void_p, c_size_t, c_void_p,
                           c_void_p, c_void_p, _P(c_int32), _P(c_int32), c_void_p]),
    "palu_fit_batch_workspace_size": (c_int32, [_P(palu_config), c_int32, c_int64, c_int32, c_int64, _P(c_size_t)]),
    "palu_fit_batch": (c_int32, [_P(palu_config), c_int32, _P(c_void_p), c_int64, c_int32, c_int64, c_void_p,
                                 c_size_t, _P(c_void_p), _P(c_void_p), _P(c_void_p), _P(c_int32), _P(c_int32),
                                 c_void_p]),
    "palu_cache_size": (c_int32, [_P(palu_config), c_int32, c_int32, c_int64, c_int32, c_int64, _P(c_size_t),
                                  _P(c_size_t), _P(c_size_t)]),
    "palu_cache_init": (c_int32, [_P(palu_cache), _P(palu_config), c_int32, c_int32, c_int64, c_int32, c_int64,
                                  c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "palu_encode_append": (c_int32, [_P(palu_cache), c_void_p, c_int64, c_void_p]),
    "palu_decode_workspace_size": (c_int32, [_P(palu_cache), _P(palu_cache), c_int32, _P(c_size_t)]),
    "palu_decode_attn": (c_int32, [_P(palu_cache), _P(palu_cache), c_void_p, c_int32, c_float, c_void_p, c_int32,
                                   c_void_p, c_size_t, c_void_p]),
    "palu_decode_attn_noalloc": (c_int32, [_P(palu_cache), _P(palu_cache), c_void_p, c_int32, c_float, c_void_p,
                                           c_int32, c_void_p]),
    "palu_decode_step": (c_int32, [_P(palu_cache), _P(palu_cache), c_void_p, c_void_p, c_void_p, c_int32, c_float,
                                   c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "palu_cache_stats": (c_int32, [_P(palu_cache), _P(palu_stats)]),
    "palu_cache_truncate": (c_int32, [_P(palu_cache), c_int64, c_void_p]),
    "palu_cache_save_size": (c_int32, [_P(palu_cache), _P(c_size_t)]),
    "palu_cache_save": (c_int32, [_P(palu_cache), c_void_p, c_size_t, c_void_p]),
    "palu_cache_restore": (c_int32, [_P(palu_cache), c_void_p, c_size_t, c_void_p]),
    "palu_cache_sync": (c_int32, [_P(palu_cache), _P(c_uint32), c_void_p]),
    "palu_debug_wait_probe": (c_int32, [_P(palu_cache), c_uint32, c_int32, c_void_p]),
    "palu_encode_append_ragged": (c_int32, [_P(palu_cache), c_void_p, c_int64, c_void_p, c_void_p]),
    "palu_cache_truncate_ragged": (c_int32, [_P(palu_cache), c_void_p, c_void_p]),
    "palu_cache_lengths": (c_int32, [_P(palu_cache), _P(c_int64), c_void_p]),
    "palu_svdq_cache_size": (c_int32, [c_int64, c_int32, _P(c_int32), c_int64, _P(c_size_t), _P(c_size_t),
                                       _P(c_size_t)]),
    "palu_svdq_cache_init": (c_int32, [_P(palu_svdq_cache), c_int64, c_int32, _P(c_int32), c_int64, c_void_p, c_int32,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "palu_svdq_append": (c_int32, [_P(palu_svdq_cache), c_void_p, c_int64, c_void_p]),
    "palu_svdq_decode_workspace_size": (c_int32, [_P(palu_svdq_cache), c_int32, _P(c_size_t)]),
    "palu_svdq_decode_attn": (c_int32, [_P(palu_svdq_cache), c_void_p, c_int64, c_void_p, c_int32, c_float, c_void_p,
                                        c_int32, c_void_p, c_size_t, c_void_p]),
    "palu_svdq_sync": (c_int32, [_P(palu_svdq_cache), _P(c_uint32), c_void_p]),
    "palu_fp16_decode_workspace_size": (c_int32, [c_int64, c_int32, c_int64, c_int32, _P(c_size_t)]),
    "palu_fp16_decode_attn": (c_int32, [c_void_p, c_void_p, c_int64, c_int32, c_int64, c_int64, c_void_p, c_int32,
                                        c_float, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "palu_kivi_cache_size": (c_int32, [c_int64, c_int32, c_int64, _P(c_size_t), _P(c_size_t)]),
    "palu_kivi_cache_init": (c_int32, [_P(palu_kivi_cache), c_int64, c_int32, c_int64, c_void_p, c_void_p]),
    "palu_kivi_append": (c_int32, [_P(palu_kivi_cache), c_void_p, c_void_p, c_int64, c_void_p]),
    "palu_kivi_decode_workspace_size": (c_int32, [_P(palu_kivi_cache), c_int32, _P(c_size_t)]),
    "palu_kivi_decode_attn": (c_int32, [_P(palu_kivi_cache), c_void_p, c_int32, c_float, c_void_p, c_int32,
                                        c_void_p, c_size_t, c_void_p]),
}

_lib = None


def lib():
    """The loaded libpalu.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpalu.so not found at {LIB_PATH}; build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


class PaluError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status):
    if status != PALU_OK:
        raise PaluError(status, lib().palu_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


_F16 = (torch.float16,)
_OUT = (torch.float32, torch.float16)
D = 128


def _need(t, name, shape, dtypes=_F16, cuda=True):
    """Refuse, before any launch, a tensor whose pointer does not describe the
    buffer the C call will read or write: the library sees the pointer only,
    so a wrong shape, type or stride would go out of bounds or read the wrong
    elements.  Entries of `shape` that are None match any extent."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.is_cuda != cuda:
        raise ValueError(f"{name} must be a {'CUDA' if cuda else 'host'} tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}; expected {' or '.join(map(str, dtypes))}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dim() != len(shape) or any(e is not None and e != s for e, s in zip(shape, t.shape)):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple('*' if e is None else e for e in shape)}")


def _dims(c):
    """(batch, kv_heads) of an initialised cache struct, else (None, None): the
    library itself reports an uninitialised cache."""
    return (c.batch, c.kv_heads) if c.magic else (None, None)


def _need_q_out(c, q, out, name="q"):
    B, _ = _dims(c)
    _need(q, name, (B, None, D))
    _need(out, "out", tuple(q.shape), _OUT)


# ------------------------------------------------------------------ entry points

def palu_last_error() -> str:
    return lib().palu_last_error().decode()


def palu_version() -> str:
    return lib().palu_version().decode()


def palu_config_default(**overrides) -> palu_config:
    cfg = palu_config()
    _check(lib().palu_config_default(ctypes.byref(cfg)))
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def palu_fit_workspace_size(cfg, batch, kv_heads, seq) -> int:
    n = c_size_t()
    _check(lib().palu_fit_workspace_size(ctypes.byref(cfg), batch, kv_heads, seq, ctypes.byref(n)))
    return n.value


def palu_fit(cfg, x, workspace, basis, mu, eigvals, stream=None):
    """x fp16 [B, Hkv, S, D] (cuda); outputs basis fp32 [n_g, D, D], mu fp32 [n_g, D],
    eigvals fp64 [n_g, D] (cuda).  Returns (rank, group_ranks)."""
    _need(x, "x", (None, None, None, D))
    B, H, S, _ = x.shape
    ng = cfg.n_head_groups
    _need(basis, "basis", (ng, D, D), (torch.float32,))
    _need(mu, "mu", (ng, D), (torch.float32,))
    _need(eigvals, "eigvals", (ng, D), (torch.float64,))
    r = c_int32()
    gr = (c_int32 * cfg.n_head_groups)()
    _check(lib().palu_fit(ctypes.byref(cfg), _ptr(x), B, H, S, _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _ptr(basis), _ptr(mu), _ptr(eigvals), ctypes.byref(r), gr, _stream(stream)))
    return r.value, list(gr)


def palu_fit_batch_workspace_size(cfgs, batch, kv_heads, seq):
    arr = (palu_config * len(cfgs))(*cfgs)
    n = c_size_t()
    _check(lib().palu_fit_batch_workspace_size(arr, len(cfgs), batch, kv_heads, seq, ctypes.byref(n)))
    return n.value


def palu_fit_batch(cfgs, xs, workspace, bases, mus, eigvals, stream=None):
    """Fit len(cfgs) tensors of one shape (xs fp16 [B, Hkv, S, D] each) in one call; outputs as
    palu_fit, per tensor.  Returns (ranks, group_ranks per tensor)."""
    n = len(cfgs)
    if n == 0 or len(xs) != n or len(bases) != n or len(mus) != n or len(eigvals) != n:
        raise ValueError("palu_fit_batch needs one tensor and one set of outputs per configuration")
    _need(xs[0], "xs[0]", (None, None, None, D))
    B, H, S, _ = xs[0].shape
    for i, c in enumerate(cfgs):
        ng = c.n_head_groups
        _need(xs[i], f"xs[{i}]", (B, H, S, D))          # one shape for every tensor
        _need(bases[i], f"bases[{i}]", (ng, D, D), (torch.float32,))
        _need(mus[i], f"mus[{i}]", (ng, D), (torch.float32,))
        _need(eigvals[i], f"eigvals[{i}]", (ng, D), (torch.float64,))
    arr = (palu_config * n)(*cfgs)
    vp = lambda ts: (c_void_p * n)(*[t.data_ptr() for t in ts])
    r = (c_int32 * n)()
    ng = [c.n_head_groups for c in cfgs]
    gr = (c_int32 * sum(ng))()
    _check(lib().palu_fit_batch(arr, n, vp(xs), B, H, S, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                vp(bases), vp(mus), vp(eigvals), r, gr, _stream(stream)))
    out, o = [], 0
    for g in ng:
        out.append(list(gr[o:o + g]))
        o += g
    return list(r), out


def palu_cache_size(cfg, role, rank, batch, kv_heads, capacity):
    a, b, c = c_size_t(), c_size_t(), c_size_t()
    _check(lib().palu_cache_size(ctypes.byref(cfg), role, rank, batch, kv_heads, capacity, ctypes.byref(a),
                                 ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def palu_cache_init(cfg, role, rank, batch, kv_heads, capacity, basis, basis_ld, mu, blocks, tail, state,
                    stream=None) -> palu_cache:
    ng = cfg.n_head_groups
    _need(basis, "basis", (ng, D, None), (torch.float32,))
    if basis_ld > basis.shape[2]:
        raise ValueError(f"basis_ld {basis_ld} exceeds the basis tensor's row length {basis.shape[2]}")
    _need(mu, "mu", (ng, D), (torch.float32,))
    c = palu_cache()
    _check(lib().palu_cache_init(ctypes.byref(c), ctypes.byref(cfg), role, rank, batch, kv_heads, capacity,
                                 _ptr(basis), basis_ld, _ptr(mu), _ptr(blocks), _ptr(tail), _ptr(state),
                                 _stream(stream)))
    return c


def palu_encode_append(cache: palu_cache, x, tokens=None, stream=None):
    """x fp16 [B, Hkv, T, D] (device); appends its T tokens (tokens, if given, must equal T)."""
    B, H = _dims(cache)
    _need(x, "x", (B, H, None, D))
    T = x.shape[2] if tokens is None else tokens
    if T != x.shape[2]:
        raise ValueError(f"tokens {T} differs from x.shape[2] = {x.shape[2]}")
    _check(lib().palu_encode_append(ctypes.byref(cache), _ptr(x), T, _stream(stream)))


def palu_decode_workspace_size(k: palu_cache, v: palu_cache, q_heads: int) -> int:
    n = c_size_t()
    _check(lib().palu_decode_workspace_size(ctypes.byref(k), ctypes.byref(v), q_heads, ctypes.byref(n)))
    return n.value


def palu_decode_attn(k, v, q, out, workspace, softmax_scale=0.0, stream=None):
    _need_q_out(k, q, out)
    _need(workspace, "workspace", (None,), (torch.uint8,))
    _check(lib().palu_decode_attn(ctypes.byref(k), ctypes.byref(v), _ptr(q), q.shape[1], softmax_scale, _ptr(out),
                                  1 if out.dtype == torch.float32 else 0, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def palu_decode_step(k, v, k_new, v_new, q, out, workspace, softmax_scale=0.0, stream=None):
    """Append one token of k and v per stream, then decode attention (k_new, v_new: [B, Hkv, D] or [B, Hkv, 1, D])."""
    B, H = _dims(k)
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, name, (B, H, D) if t.dim() == 3 else (B, H, 1, D))
    _need_q_out(k, q, out)
    _need(workspace, "workspace", (None,), (torch.uint8,))
    _check(lib().palu_decode_step(ctypes.byref(k), ctypes.byref(v), _ptr(k_new), _ptr(v_new), _ptr(q), q.shape[1],
                                  softmax_scale, _ptr(out), 1 if out.dtype == torch.float32 else 0, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def palu_decode_attn_noalloc(k, v, q, out, softmax_scale=0.0, stream=None):
    """palu_decode_attn using the library's fixed device scratch (no workspace)."""
    _need_q_out(k, q, out)
    _check(lib().palu_decode_attn_noalloc(ctypes.byref(k), ctypes.byref(v), _ptr(q), q.shape[1], softmax_scale,
                                          _ptr(out), 1 if out.dtype == torch.float32 else 0, _stream(stream)))


def palu_cache_stats(cache) -> dict:
    s = palu_stats()
    _check(lib().palu_cache_stats(ctypes.byref(cache), ctypes.byref(s)))
    return {name: getattr(s, name) for name, _ in palu_stats._fields_}


def palu_cache_truncate(cache, length, stream=None):
    _check(lib().palu_cache_truncate(ctypes.byref(cache), length, _stream(stream)))


def palu_cache_save_size(cache) -> int:
    n = c_size_t()
    _check(lib().palu_cache_save_size(ctypes.byref(cache), ctypes.byref(n)))
    return n.value


def palu_cache_save(cache, host, stream=None):
    """Copy the cache image into `host` (a CPU uint8 tensor of >= palu_cache_save_size bytes)."""
    _need(host, "host", (None,), (torch.uint8,), cuda=False)
    _check(lib().palu_cache_save(ctypes.byref(cache), c_void_p(host.data_ptr()), host.numel(), _stream(stream)))


def palu_cache_restore(cache, host, stream=None):
    """Copy a cache image (a CPU uint8 tensor) into `cache`."""
    _need(host, "host", (None,), (torch.uint8,), cuda=False)
    _check(lib().palu_cache_restore(ctypes.byref(cache), c_void_p(host.data_ptr()), host.numel(), _stream(stream)))


def palu_cache_sync(cache, stream=None) -> int:
    """Synchronise and refresh cache.length; raises PaluError if the device error word was set."""
    e = c_uint32()
    _check(lib().palu_cache_sync(ctypes.byref(cache), ctypes.byref(e), _stream(stream)))
    return e.value


def palu_encode_append_ragged(cache: palu_cache, x, counts, stream=None):
    """x [B, Hkv, T, D] fp16 (device); counts int32 [B] (device): sequence b appends its first counts[b] rows."""
    B, H = _dims(cache)
    _need(x, "x", (B, H, None, D))
    _need(counts, "counts", (B,), (torch.int32,))
    _check(lib().palu_encode_append_ragged(ctypes.byref(cache), _ptr(x), x.shape[2], _ptr(counts), _stream(stream)))


def palu_cache_truncate_ragged(cache: palu_cache, lengths, stream=None):
    """lengths int64 [B] (device): per-sequence rollback."""
    _need(lengths, "lengths", (_dims(cache)[0],), (torch.int64,))
    _check(lib().palu_cache_truncate_ragged(ctypes.byref(cache), _ptr(lengths), _stream(stream)))


def palu_cache_lengths(cache: palu_cache, stream=None) -> list:
    """Each sequence's length (synchronises)."""
    out = (c_int64 * cache.batch)()
    _check(lib().palu_cache_lengths(ctypes.byref(cache), out, _stream(stream)))
    return list(out)


def palu_debug_wait_probe(cache, spin_limit, signal, stream=None):
    """Run the library's bounded wait on a barrier that is signalled or left pending."""
    _check(lib().palu_debug_wait_probe(ctypes.byref(cache), spin_limit, 1 if signal else 0, _stream(stream)))


def palu_fp16_decode_workspace_size(batch, kv_heads, seq_cap, q_heads) -> int:
    n = c_size_t()
    _check(lib().palu_fp16_decode_workspace_size(batch, kv_heads, seq_cap, q_heads, ctypes.byref(n)))
    return n.value


def palu_fp16_decode_attn(k, v, seq, q, out, workspace, softmax_scale=0.0, stream=None):
    """k, v fp16 [B, Hkv, cap, D] (tokens 0..seq-1 used), q fp16 [B, Hq, D], out [B, Hq, D] (device)."""
    _need(k, "k", (None, None, None, D))
    B, H, cap, _ = k.shape
    _need(v, "v", (B, H, cap, D))
    _need(q, "q", (B, None, D))
    _need(out, "out", tuple(q.shape), _OUT)
    _need(workspace, "workspace", (None,), (torch.uint8,))
    _check(lib().palu_fp16_decode_attn(_ptr(k), _ptr(v), B, H, seq, cap, _ptr(q), q.shape[1], softmax_scale,
                                       _ptr(out), 1 if out.dtype == torch.float32 else 0, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def palu_kivi_cache_size(batch, kv_heads, capacity):
    r, w = c_size_t(), c_size_t()
    _check(lib().palu_kivi_cache_size(batch, kv_heads, capacity, ctypes.byref(r), ctypes.byref(w)))
    return r.value, w.value


def palu_kivi_cache_init(batch, kv_heads, capacity, records, window) -> palu_kivi_cache:
    c = palu_kivi_cache()
    _check(lib().palu_kivi_cache_init(ctypes.byref(c), batch, kv_heads, capacity, _ptr(records), _ptr(window)))
    return c


def palu_kivi_append(cache: palu_kivi_cache, k, v, tokens=None, stream=None):
    """k, v fp16 [B, Hkv, T, D] (device); appends their T tokens (tokens, if given, must equal T)."""
    B, H = _dims(cache)
    _need(k, "k", (B, H, None, D))
    _need(v, "v", tuple(k.shape))
    n = k.shape[2] if tokens is None else tokens
    if n != k.shape[2]:
        raise ValueError(f"tokens {n} differs from k.shape[2] = {k.shape[2]}")
    _check(lib().palu_kivi_append(ctypes.byref(cache), _ptr(k), _ptr(v), n, _stream(stream)))


def palu_kivi_decode_workspace_size(cache: palu_kivi_cache, q_heads: int) -> int:
    n = c_size_t()
    _check(lib().palu_kivi_decode_workspace_size(ctypes.byref(cache), q_heads, ctypes.byref(n)))
    return n.value


def palu_kivi_decode_attn(cache: palu_kivi_cache, q, out, workspace, softmax_scale=0.0, stream=None):
    _need_q_out(cache, q, out)
    _need(workspace, "workspace", (None,), (torch.uint8,))
    _check(lib().palu_kivi_decode_attn(ctypes.byref(cache), _ptr(q), q.shape[1], softmax_scale, _ptr(out),
                                       1 if out.dtype == torch.float32 else 0, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


# ------------------------------------------------------------------ buffer helpers

def _dev_bytes(n, device):
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


class LatentCache:
    """One (layer, K or V) cache with its device buffers allocated by torch."""

    def __init__(self, cfg, role, rank, batch, kv_heads, capacity, basis, mu, basis_ld=None, stream=None):
        dev = basis.device
        blk, tail, state = palu_cache_size(cfg, role, rank, batch, kv_heads, capacity)
        self.blocks = _dev_bytes(blk, dev)
        self.tail = _dev_bytes(tail, dev) if tail else None
        self.state = _dev_bytes(state, dev)
        ld = basis.shape[-1] if basis_ld is None else basis_ld
        self.c = palu_cache_init(cfg, role, rank, batch, kv_heads, capacity, basis, ld, mu, self.blocks,
                                 self.tail, self.state, stream)

    @property
    def length(self):
        return self.c.length

    def append(self, x, stream=None):
        palu_encode_append(self.c, x, x.shape[2], stream)

    def stats(self):
        return palu_cache_stats(self.c)

    def sync(self, stream=None):
        return palu_cache_sync(self.c, stream)

    def truncate(self, length, stream=None):
        palu_cache_truncate(self.c, length, stream)

    def append_ragged(self, x, counts, stream=None):
        """Sequence b appends its first counts[b] rows of x (counts: int32 tensor on the device)."""
        palu_encode_append_ragged(self.c, x, counts, stream)

    def truncate_ragged(self, lengths, stream=None):
        palu_cache_truncate_ragged(self.c, lengths, stream)

    def lengths(self, stream=None):
        return palu_cache_lengths(self.c, stream)

    def save(self, stream=None):
        """The cache image in pinned host memory (complete once `stream` has passed the call)."""
        host = torch.empty(palu_cache_save_size(self.c), dtype=torch.uint8, pin_memory=torch.cuda.is_available())
        palu_cache_save(self.c, host, stream)
        return host

    def restore(self, image, stream=None):
        palu_cache_restore(self.c, image, stream)

    def record_array(self):
        """Block records as a host uint8 array [B, Hkv, n_blk_cap, record_bytes]."""
        c = self.c
        n = c.batch * c.kv_heads * c.n_blk_cap * c.record_bytes
        return self.blocks[:n].cpu().numpy().reshape(c.batch, c.kv_heads, c.n_blk_cap, c.record_bytes)

    def tail_array(self):
        c = self.c
        if self.tail is None:
            return None
        n = c.batch * c.kv_heads * 32 * c.rank * 4
        return self.tail[:n].cpu().numpy().view("float32").reshape(c.batch, c.kv_heads, 32, c.rank)

    def basis_array(self):
        """The stored basis as [n_g, D, r] and mean [n_g, D] (host fp32)."""
        c = self.c
        ng, r = c.n_groups, c.rank
        st = self.state.cpu().numpy()
        basis_off = 256
        mu_off = -(-(basis_off + 4 * ng * r * 128) // 256) * 256
        bT = st[basis_off:basis_off + 4 * ng * r * 128].view("float32").reshape(ng, r, 128)
        mu = st[mu_off:mu_off + 4 * ng * 128].view("float32").reshape(ng, 128)
        return bT.transpose(0, 2, 1).copy(), mu.copy()


class KiviCache:
    """A KIVI-2bit cache of one layer (keys and values) with torch-allocated buffers."""

    def __init__(self, batch, kv_heads, capacity, device):
        rec, win = palu_kivi_cache_size(batch, kv_heads, capacity)
        self.records = _dev_bytes(rec, device)
        self.window = _dev_bytes(win, device)
        self.c = palu_kivi_cache_init(batch, kv_heads, capacity, self.records, self.window)

    @property
    def length(self):
        return self.c.length

    def append(self, k, v, stream=None):
        palu_kivi_append(self.c, k, v, k.shape[2], stream)

    def decode(self, q, out_dtype=torch.float32, softmax_scale=0.0, stream=None, workspace=None, out=None):
        if workspace is None:
            workspace = _dev_bytes(palu_kivi_decode_workspace_size(self.c, q.shape[1]), q.device)
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
        palu_kivi_decode_attn(self.c, q, out, workspace, softmax_scale, stream)
        return out

    def record_array(self):
        """Block records as a host uint8 array [B, Hkv, n_blk_cap, 3072]."""
        c = self.c
        n = c.batch * c.kv_heads * c.n_blk_cap * 3072
        return self.records[:n].cpu().numpy().reshape(c.batch, c.kv_heads, c.n_blk_cap, 3072)

    def window_array(self):
        """The window as host fp16 [B, Hkv, 2 (keys, values), 32, 128]."""
        c = self.c
        n = c.batch * c.kv_heads * 2 * 32 * 128 * 2
        return self.window[:n].cpu().numpy().view("float16").reshape(c.batch, c.kv_heads, 2, 32, 128)


class SvdqCache:
    """An SVDq keys-only cache of one layer (include/svdq.h) with torch-allocated buffers.
    ranks: per-head ranks; basis fp32 [Hkv, D, ld] and mu [Hkv, D] on the device (palu_fit with one head per group)."""

    def __init__(self, batch, kv_heads, ranks, capacity, basis, mu, stream=None):
        dev = basis.device
        if len(ranks) != kv_heads:
            raise ValueError(f"{len(ranks)} ranks given for {kv_heads} KV heads")
        _need(basis, "basis", (kv_heads, D, None), (torch.float32,))
        _need(mu, "mu", (kv_heads, D), (torch.float32,))
        rk = (c_int32 * kv_heads)(*[int(r) for r in ranks])
        bb, tb, sb = c_size_t(), c_size_t(), c_size_t()
        _check(lib().palu_svdq_cache_size(batch, kv_heads, rk, capacity, ctypes.byref(bb), ctypes.byref(tb),
                                          ctypes.byref(sb)))
        self.blocks = _dev_bytes(bb.value, dev)
        self.tail = _dev_bytes(tb.value, dev)
        self.state = _dev_bytes(sb.value, dev)
        self.ranks = [int(r) for r in ranks]
        self.c = palu_svdq_cache()
        _check(lib().palu_svdq_cache_init(ctypes.byref(self.c), batch, kv_heads, rk, capacity, _ptr(basis),
                                          basis.shape[-1], _ptr(mu), _ptr(self.blocks), _ptr(self.tail),
                                          _ptr(self.state), _stream(stream)))

    @property
    def length(self):
        return self.c.length

    def append(self, k, stream=None):
        """k fp16 [B, Hkv, T, D] on the device."""
        _need(k, "k", (*_dims(self.c), None, D))
        _check(lib().palu_svdq_append(ctypes.byref(self.c), _ptr(k), k.shape[2], _stream(stream)))

    def decode(self, v, q, out_dtype=torch.float32, softmax_scale=0.0, stream=None, workspace=None, out=None):
        """v fp16 [B, Hkv, v_cap, D] (tokens 0..length-1 used), q fp16 [B, Hq, D]; returns out [B, Hq, D]."""
        _need(v, "v", (*_dims(self.c), None, D))
        _need(q, "q", (_dims(self.c)[0], None, D))
        if workspace is None:
            n = c_size_t()
            _check(lib().palu_svdq_decode_workspace_size(ctypes.byref(self.c), q.shape[1], ctypes.byref(n)))
            workspace = _dev_bytes(n.value, q.device)
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
        _need(out, "out", tuple(q.shape), _OUT)
        _need(workspace, "workspace", (None,), (torch.uint8,))
        _check(lib().palu_svdq_decode_attn(ctypes.byref(self.c), _ptr(v), v.shape[2], _ptr(q), q.shape[1],
                                           c_float(softmax_scale), _ptr(out), 1 if out.dtype == torch.float32 else 0,
                                           _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def sync(self, stream=None):
        e = c_uint32()
        _check(lib().palu_svdq_sync(ctypes.byref(self.c), ctypes.byref(e), _stream(stream)))
        return e.value

    def record_array(self):
        """Block records as a host uint8 array [B, Hkv, n_blk_cap, record_bytes]."""
        c = self.c
        n = c.batch * c.kv_heads * c.n_blk_cap * c.record_bytes
        return self.blocks[:n].cpu().numpy().reshape(c.batch, c.kv_heads, c.n_blk_cap, c.record_bytes)

    def tail_array(self):
        """The fp32 tail latents [B, Hkv, 32, r_max] (host)."""
        c = self.c
        n = c.batch * c.kv_heads * 32 * c.r_max * 4
        return self.tail[:n].cpu().numpy().view("float32").reshape(c.batch, c.kv_heads, 32, c.r_max)


def fit(cfg, x, stream=None):
    """Run palu_fit on x fp16 [B, Hkv, S, D]; returns (basis, mu, eigvals, rank, group_ranks)."""
    B, H, S, D = x.shape
    ng = cfg.n_head_groups
    ws = _dev_bytes(palu_fit_workspace_size(cfg, B, H, S), x.device)
    basis = torch.empty(ng, D, D, dtype=torch.float32, device=x.device)
    mu = torch.empty(ng, D, dtype=torch.float32, device=x.device)
    eig = torch.empty(ng, D, dtype=torch.float64, device=x.device)
    r, gr = palu_fit(cfg, x, ws, basis, mu, eig, stream)
    return basis, mu, eig, r, gr


def fit_batch(cfgs, xs, stream=None):
    """Run palu_fit_batch on tensors xs (fp16 [B, Hkv, S, D], one shape) with configurations cfgs;
    returns [(basis, mu, eigvals, rank, group_ranks)] per tensor."""
    B, H, S, D = xs[0].shape
    if any(tuple(x.shape) != tuple(xs[0].shape) for x in xs):
        raise ValueError("fit_batch needs tensors of one shape")
    dev = xs[0].device
    ws = _dev_bytes(palu_fit_batch_workspace_size(cfgs, B, H, S), dev)
    bases = [torch.empty(c.n_head_groups, D, D, dtype=torch.float32, device=dev) for c in cfgs]
    mus = [torch.empty(c.n_head_groups, D, dtype=torch.float32, device=dev) for c in cfgs]
    eigs = [torch.empty(c.n_head_groups, D, dtype=torch.float64, device=dev) for c in cfgs]
    ranks, grs = palu_fit_batch(cfgs, xs, ws, bases, mus, eigs, stream)
    return [(bases[i], mus[i], eigs[i], ranks[i], grs[i]) for i in range(len(cfgs))]


def decode(kc: LatentCache, vc: LatentCache, q, out_dtype=torch.float32, softmax_scale=0.0, stream=None,
           workspace=None, out=None):
    """Decode attention; returns out [B, Hq, D]."""
    if workspace is None:
        workspace = _dev_bytes(palu_decode_workspace_size(kc.c, vc.c, q.shape[1]), q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    palu_decode_attn(kc.c, vc.c, q, out, workspace, softmax_scale, stream)
    return out


def decode_step(kc: LatentCache, vc: LatentCache, k_new, v_new, q, out_dtype=torch.float32, softmax_scale=0.0,
                stream=None, workspace=None, out=None):
    """One decode step: append k_new, v_new ([B, Hkv, 1, D] fp16), then decode attention; returns out."""
    if workspace is None:
        workspace = _dev_bytes(palu_decode_workspace_size(kc.c, vc.c, q.shape[1]), q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    palu_decode_step(kc.c, vc.c, k_new, v_new, q, out, workspace, softmax_scale, stream)
    return out
