"""GB300-native group-head low-rank latent KV cache (PALU style).

The compute path is the C-ABI library libpalu.so (hand-written CUDA for
sm_103a); `rank_latent_kv_gb300.palu` is its thin ctypes binding.
"""
