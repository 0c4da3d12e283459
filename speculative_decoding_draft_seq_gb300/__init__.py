"""DSpark per-round draft -> schedule -> verify hot path for one GB300 (sm_103a).

The compute lives in libdspark.so (CUDA kernels behind the C ABI of
include/dspark.h); `speculative_decoding_draft_seq_gb300.dspark` is its Python
binding. Import the binding explicitly; importing this package alone loads
nothing.
"""
__all__ = ["dspark", "build"]
