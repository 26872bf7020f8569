"""GB300-native compressed sparse attention forward (window ring + compressed
latent rows + fp4 indexer top-k + sparse attention with a per-head sink).

The compute lives in ``libds41.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/ds41.h``); :mod:`.ds41` is the thin ctypes binding
that marshals torch tensors into that ABI.  :mod:`.workloads` holds the
workload shapes and the seeded synthetic input generator.
"""
__all__ = ["ds41", "workloads"]
