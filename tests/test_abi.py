"""The C-ABI library loads, exports every symbol declared in include/*.h,
its structs match the binding's, and host-side validation works (no GPU)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest
import torch

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "palu.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))


@pytest.fixture(scope="session")
def palu():
    from rank_latent_kv_gb300 import palu as P
    if not os.path.exists(P.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    P.lib()
    return P


def declared_functions():
    src = "".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(palu_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("palu_fit", "palu_encode_append", "palu_decode_attn", "palu_cache_init", "palu_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(palu):
    out = subprocess.run(["nm", "-D", "--defined-only", palu.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (palu_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(palu.lib(), n)
    assert set(palu._SIGNATURES) == set(declared_functions())


def test_struct_layouts_match_the_header(palu):
    """Compile a tiny C program against palu.h and compare sizes/offsets with ctypes."""
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "palu.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(palu_config), sizeof(palu_cache), sizeof(palu_stats),
         offsetof(palu_config, energy_threshold), offsetof(palu_cache, capacity), offsetof(palu_cache, length),
         offsetof(palu_stats, code_bytes));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        vals = list(map(int, subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()))
    assert vals == [ctypes.sizeof(palu.palu_config), ctypes.sizeof(palu.palu_cache), ctypes.sizeof(palu.palu_stats),
                    palu.palu_config.energy_threshold.offset, palu.palu_cache.capacity.offset,
                    palu.palu_cache.length.offset, palu.palu_stats.code_bytes.offset]


def test_defaults_follow_the_page(palu):
    cfg = palu.palu_config_default()
    assert (cfg.head_dim, cfg.n_head_groups, cfg.rank, cfg.hi_bit, cfg.lo_bit, cfg.group_size, cfg.quantize) == \
           (128, 4, 0, 4, 2, 32, 1)
    assert cfg.energy_threshold == 0.90 and cfg.hi_fraction == 0.25
    assert "sm_103a" in palu.palu_version()


def test_cache_size_matches_the_layout(palu):
    import oracle as O
    cfg = palu.palu_config_default()
    for role in (palu.PALU_ROLE_KEY, palu.PALU_ROLE_VALUE):
        for r in (1, 27, 32, 52, 74, 128):
            blk, tail, state = palu.palu_cache_size(cfg, role, r, 2, 8, 100)
            rec = O.Layout(role, r, O.n_hi_channels(r)).record_bytes
            assert blk == -(-(2 * 8 * 4 * rec) // 256) * 256
            assert tail == -(-(4 * 2 * 8 * 32 * r) // 256) * 256
            assert state % 256 == 0 and state >= 4 * 4 * r * 128
    cfg.quantize = 0
    blk, tail, _ = palu.palu_cache_size(cfg, palu.PALU_ROLE_VALUE, 32, 1, 8, 64)
    assert blk == 8 * 2 * 4 * 512 and tail == 0


@pytest.mark.parametrize("change,status", [
    (dict(head_dim=64), 2), (dict(group_size=16), 2), (dict(hi_bit=8), 2), (dict(n_head_groups=3), 1),
    (dict(hi_fraction=1.5), 1)])
def test_host_validation_errors(palu, change, status):
    cfg = palu.palu_config_default(**change)
    with pytest.raises(palu.PaluError) as e:
        palu.palu_cache_size(cfg, palu.PALU_ROLE_KEY, 32, 1, 8, 64)
    assert e.value.status == status
    assert palu.palu_last_error()


def test_rank_and_role_validation(palu):
    cfg = palu.palu_config_default()
    for bad in (0, 129):
        with pytest.raises(palu.PaluError):
            palu.palu_cache_size(cfg, palu.PALU_ROLE_KEY, bad, 1, 8, 64)
    cfg.quantize = 0
    with pytest.raises(palu.PaluError) as e:
        palu.palu_cache_size(cfg, palu.PALU_ROLE_KEY, 32, 1, 8, 64)
    assert "value caches only" in str(e.value)


def test_fit_workspace_and_validation(palu):
    cfg = palu.palu_config_default()
    n = palu.palu_fit_workspace_size(cfg, 1, 8, 4096)
    assert n >= 4 * 2 * 128 * 128 * 4 + 4 * 128 * 128 * 8     # >= one (hi, lo) chunk per group + fp64 Gram
    with pytest.raises(palu.PaluError):
        palu.palu_fit_workspace_size(palu.palu_config_default(energy_threshold=0.0), 1, 8, 64)
    with pytest.raises(palu.PaluError):
        palu.palu_fit_workspace_size(cfg, 1, 6, 64)


def test_cache_image_calls_reject_uninitialised_caches(palu):
    c = palu.palu_cache()
    n = ctypes.c_size_t()
    assert palu.lib().palu_cache_save_size(ctypes.byref(c), ctypes.byref(n)) == 4
    buf = (ctypes.c_uint8 * 256)()
    assert palu.lib().palu_cache_save(ctypes.byref(c), buf, 256, None) == 4
    assert palu.lib().palu_cache_restore(ctypes.byref(c), buf, 256, None) == 4
    assert "not initialised" in palu.palu_last_error()


def test_uninitialised_cache_is_rejected(palu):
    c = palu.palu_cache()
    st = palu.palu_stats()
    assert palu.lib().palu_cache_stats(ctypes.byref(c), ctypes.byref(st)) == 4
    assert "not initialised" in palu.palu_last_error()


def test_fp16_comparator_validation(palu):
    with pytest.raises(palu.PaluError):
        palu.palu_fp16_decode_workspace_size(1, 4, 128, 40)   # 10 query heads per KV head


def test_kivi_struct_layout_and_sizes(palu):
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "kivi.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(palu_kivi_cache), offsetof(palu_kivi_cache, capacity),
         offsetof(palu_kivi_cache, records), offsetof(palu_kivi_cache, length));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        vals = list(map(int, subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()))
    K = palu.palu_kivi_cache
    assert vals == [ctypes.sizeof(K), K.capacity.offset, K.records.offset, K.length.offset]
    from oracle import kivi_oracle
    # records: one 3072-byte record per complete block; window: 2 x 32 x 128 fp16 per stream
    rec, win = palu.palu_kivi_cache_size(3, 4, 32 * 10 + 17)
    assert rec == -(-(12 * 10 * kivi_oracle.RECORD) // 256) * 256 and win == 12 * 2 * 32 * 128 * 2


def test_kivi_host_validation(palu):
    """Errors the host detects without launching anything (fake, aligned device addresses)."""
    c = palu.palu_kivi_cache()
    with pytest.raises(palu.PaluError) as e:
        palu._check(palu.lib().palu_kivi_append(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), 1, None))
    assert e.value.status == 4  # not initialised
    c = palu.palu_kivi_cache_init(2, 2, 100, torch_like(1 << 20), torch_like(1 << 21))
    assert (c.length, c.n_blk_cap, c.bits) == (0, 3, 2)
    with pytest.raises(palu.PaluError) as e:
        palu._check(palu.lib().palu_kivi_append(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), 101,
                                                None))
    assert e.value.status == 3  # capacity
    with pytest.raises(palu.PaluError) as e:
        palu._check(palu.lib().palu_kivi_append(ctypes.byref(c), ctypes.c_void_p(8), ctypes.c_void_p(256), 1, None))
    assert e.value.status == 1  # misaligned
    assert palu.lib().palu_kivi_append(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), 0, None) == 0
    n = ctypes.c_size_t()
    assert palu.lib().palu_kivi_decode_workspace_size(ctypes.byref(c), 3, ctypes.byref(n)) == 1   # 3 % 2
    assert palu.lib().palu_kivi_decode_workspace_size(ctypes.byref(c), 18, ctypes.byref(n)) == 2  # 9 per KV head
    # decoding an empty cache
    assert palu.lib().palu_kivi_decode_attn(ctypes.byref(c), ctypes.c_void_p(256), 2, 0.0, ctypes.c_void_p(256), 1,
                                            ctypes.c_void_p(256), 1 << 20, None) == 1
    for bad in ((0, 2, 10), (1, 0, 10), (1, 2, 0)):
        with pytest.raises(palu.PaluError):
            palu.palu_kivi_cache_size(*bad)


class torch_like:
    """An object with a data_ptr() for the binding's pointer marshalling (never dereferenced)."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def test_svdq_struct_layout_and_sizes(palu):
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "svdq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(palu_svdq_cache), offsetof(palu_svdq_cache, capacity),
         offsetof(palu_svdq_cache, blocks), offsetof(palu_svdq_cache, state), offsetof(palu_svdq_cache, length));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        vals = list(map(int, subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()))
    C = palu.palu_svdq_cache
    assert vals == [ctypes.sizeof(C), C.capacity.offset, C.blocks.offset, C.state.offset, C.length.offset]
    # record stride: the largest head's record (the oracle's layout), 16-byte multiple; tail: 32 x r_max fp32
    from oracle import svdq_oracle as S
    ranks = [1, 74, 128, 7]
    rk = (ctypes.c_int32 * 4)(*ranks)
    bb, tb, sb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    palu._check(palu.lib().palu_svdq_cache_size(3, 4, rk, 100, ctypes.byref(bb), ctypes.byref(tb), ctypes.byref(sb)))
    stride = max(S.record_layout(r)[4] for r in ranks)
    assert bb.value == -(-(3 * 4 * 4 * stride) // 256) * 256
    assert tb.value == -(-(3 * 4 * 32 * 128 * 4) // 256) * 256
    assert sb.value > 4 * 128 * 128 * 4  # holds the transposed bases


def test_svdq_host_validation(palu):
    """Errors the host detects before any launch."""
    bb, tb, sb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    for ranks in ([0, 8], [8, 129]):
        rk = (ctypes.c_int32 * 2)(*ranks)
        assert palu.lib().palu_svdq_cache_size(1, 2, rk, 64, ctypes.byref(bb), ctypes.byref(tb), ctypes.byref(sb)) == 1
    rk = (ctypes.c_int32 * 2)(8, 16)
    assert palu.lib().palu_svdq_cache_size(0, 2, rk, 64, ctypes.byref(bb), ctypes.byref(tb), ctypes.byref(sb)) == 1
    assert palu.lib().palu_svdq_cache_size(1, 2, None, 64, ctypes.byref(bb), ctypes.byref(tb), ctypes.byref(sb)) == 1
    c = palu.palu_svdq_cache()
    a = ctypes.c_void_p(1 << 20)
    # misaligned buffers, a NULL basis, and a basis row stride below the largest rank
    assert palu.lib().palu_svdq_cache_init(ctypes.byref(c), 1, 2, rk, 64, a, 128, a, ctypes.c_void_p(16), a, a,
                                           None) == 1
    assert palu.lib().palu_svdq_cache_init(ctypes.byref(c), 1, 2, rk, 64, None, 128, a, a, a, a, None) == 1
    assert palu.lib().palu_svdq_cache_init(ctypes.byref(c), 1, 2, rk, 64, a, 8, a, a, a, a, None) == 1
    # an uninitialised cache
    n = ctypes.c_size_t()
    assert palu.lib().palu_svdq_decode_workspace_size(ctypes.byref(c), 4, ctypes.byref(n)) == 4
    assert palu.lib().palu_svdq_append(ctypes.byref(c), a, 1, None) == 4
    assert "not initialised" in palu.palu_last_error()


def test_fit_batch_workspace_and_validation(palu):
    cfg = palu.palu_config_default(n_head_groups=2)
    one = palu.palu_fit_workspace_size(cfg, 2, 4, 4096)
    assert palu.palu_fit_batch_workspace_size([cfg], 2, 4, 4096) == one
    two = palu.palu_fit_batch_workspace_size([cfg, cfg], 2, 4, 4096)
    # the partial-sum area is shared: a second tensor adds only its fp64 Gram matrices and error word
    assert two - one == 2 * 128 * 128 * 8 + 256
    with pytest.raises(palu.PaluError):
        palu.palu_fit_batch_workspace_size([cfg, palu.palu_config_default(n_head_groups=3)], 2, 4, 4096)
    arr = (palu.palu_config * 1)(cfg)
    n = ctypes.c_size_t()
    assert palu.lib().palu_fit_batch_workspace_size(arr, 0, 2, 4, 4096, ctypes.byref(n)) == 1
    r = (ctypes.c_int32 * 1)()
    assert palu.lib().palu_fit_batch(arr, 1, None, 2, 4, 4096, ctypes.c_void_p(1 << 20), 1 << 30, None, None, None,
                                     r, None, None) == 1


def test_binding_refuses_tensors_before_any_call(palu):
    """The binding checks every tensor whose pointer crosses the C ABI (the
    library sees the pointer only): device, dtype, contiguity and shape."""
    x = torch.zeros(2, 3, 5, 128, dtype=torch.float16)
    palu._need(x, "x", (2, 3, None, 128), cuda=False)
    for bad in (x.float(), x.transpose(1, 2), x[:, :2], x[..., :64]):
        with pytest.raises(ValueError):
            palu._need(bad, "x", (2, 3, None, 128), cuda=False)
    with pytest.raises(ValueError):
        palu._need(x, "x", (2, 3, None, 128))                     # a host tensor where the device is needed
    with pytest.raises(ValueError):
        palu._need(x.reshape(6, 5, 128), "x", (2, 3, None, 128), cuda=False)
    with pytest.raises(ValueError):
        palu._need(torch_like(256), "x", (None,), cuda=False)
    # the wrappers run the checks before they call the library (host tensors here)
    c = palu.palu_cache()
    q = torch.zeros(1, 4, 128, dtype=torch.float16)
    ws = torch.zeros(256, dtype=torch.uint8)
    for call in (lambda: palu.palu_decode_attn(c, c, q, q, ws),
                 lambda: palu.palu_decode_attn_noalloc(c, c, q, q),
                 lambda: palu.palu_encode_append(c, x),
                 lambda: palu.palu_fp16_decode_attn(x, x, 5, q, q, ws),
                 lambda: palu.palu_kivi_decode_attn(palu.palu_kivi_cache(), q, q, ws),
                 lambda: palu.palu_cache_save(c, torch_like(256))):
        with pytest.raises(ValueError):
            call()
