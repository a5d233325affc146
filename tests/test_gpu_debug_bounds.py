"""The bounds-checking build (libpalu_debug.so, compiled with
-DPALU_DEBUG_BOUNDS=1).  Its encode record writes, one-token appends (the
latent cache's, also inside the fused decode step) and SVDq record writes
check their block indices against the cache and would report
PALU_DEVERR_BOUNDS instead of writing out of range.  On valid calls it reports
nothing, and every result equals the default build's bit for bit.  The debug
library runs in a child process (a process loads one library).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_case(P, out_path):
    """Fit, prefill, fused decode steps across block boundaries, a decode, and
    an SVDq cache; saves the outputs and returns the caches' error words."""
    dev = "cuda"
    rng = np.random.default_rng(77)
    B, H, Hq, S, steps = 2, 4, 8, 100, 30
    x = rng.standard_normal((2, B, H, S + steps, 128)).astype(np.float16)
    q = torch.from_numpy(rng.standard_normal((steps + 1, B, Hq, 128)).astype(np.float16)).to(dev)
    caches = []
    for t, (role, rank) in enumerate(((P.PALU_ROLE_KEY, 24), (P.PALU_ROLE_VALUE, 48))):
        xt = torch.from_numpy(x[t, :, :, :S].copy()).to(dev)
        cfg = P.palu_config_default(n_head_groups=2, rank=rank)
        basis, mu, _, _, _ = P.fit(cfg, xt)
        c = P.LatentCache(cfg, role, rank, B, H, S + steps + 8, basis, mu)
        c.append(xt)
        caches.append(c)
    kc, vc = caches
    outs = []
    for i in range(steps):
        kn = torch.from_numpy(x[0, :, :, S + i].copy()).to(dev)
        vn = torch.from_numpy(x[1, :, :, S + i].copy()).to(dev)
        outs.append(P.decode_step(kc, vc, kn, vn, q[i]))
    outs.append(P.decode(kc, vc, q[steps]))
    # SVDq keys: per-head fit, prefill, one-token appends, decode with fp16 values
    k = torch.from_numpy(x[0].copy()).to(dev)
    cfg = P.palu_config_default(n_head_groups=H, rank=0, energy_threshold=0.95)
    basis, mu, _, _, gr = P.fit(cfg, k[:, :, :S].contiguous())
    sc = P.SvdqCache(B, H, gr, S + steps, basis, mu)
    sc.append(k[:, :, :S].contiguous())
    for i in range(3):
        sc.append(k[:, :, S + i:S + i + 1].contiguous())
    v = torch.from_numpy(x[1].copy()).to(dev)
    outs.append(sc.decode(v, q[0]))
    torch.cuda.synchronize()
    np.save(out_path, torch.stack([o.float() for o in outs]).cpu().numpy())
    return [kc.sync(), vc.sync(), sc.sync()]


CHILD = r"""
import sys
sys.path.insert(0, {root!r})
from rank_latent_kv_gb300 import palu as P
P.LIB_PATH = {lib!r}
import tests.test_gpu_debug_bounds as T
print("ERR", *T.run_case(P, {out!r}))
"""


def test_debug_bounds_build_reports_nothing_and_matches(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rank_latent_kv_gb300 import build, palu as P
    lib = build.LIB_DEBUG
    if not os.path.exists(lib):
        build.build(debug_bounds=True)
    out_dbg = str(tmp_path / "debug.npy")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=lib, out=out_dbg)],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    errs = [int(v) for v in r.stdout.split("ERR", 1)[1].split()]
    assert errs == [0, 0, 0], f"device error words of the debug build: {errs}"
    P.lib()
    out_def = str(tmp_path / "default.npy")
    assert run_case(P, out_def) == [0, 0, 0]
    a, b = np.load(out_dbg), np.load(out_def)
    assert np.isfinite(a).all() and np.array_equal(a, b)
