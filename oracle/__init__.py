"""CPU oracle for the group-head low-rank latent KV cache, for the KIVI-2bit
cache it is compared with (oracle.kivi_oracle), for the SVDq keys-only
variant (oracle.svdq_oracle) and for ragged per-sequence lengths
(oracle.ragged_oracle).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the method computes, written from the method's
description (PALU — True Low-Rank Latent Storage for Keys and Values; the
SVDq cache module page; the KIVI quantizer and bit-packing passages of the
VeloxQuant-MLX blog).  It is used by the tests, by the package's smoke check
and by the benchmark's CPU-baseline leg.  The product path never imports it,
and it shares no code with the CUDA path.

Every function pinned by a test against something other than itself (closed
forms, constructed spectra, library routines, hand-worked cases).  See
tests/test_oracle_pins.py, tests/test_kivi_oracle_pins.py,
tests/test_svdq_oracle_pins.py and tests/test_ragged_oracle_pins.py.
"""
from .palu_oracle import *  # noqa: F401,F403
from . import kivi_oracle  # noqa: F401
from . import svdq_oracle  # noqa: F401
from . import ragged_oracle  # noqa: F401
