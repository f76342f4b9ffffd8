"""GB300-native ZeRO-DP partitioned mixed-precision AdamW step.

One GPU holds N_d simulated data-parallel ranks as separate HBM buffers.  The
step reduce-scatters the ranks' 16-bit gradient replicas over a flat, padded,
bucketed buffer, computes a sharding-aware global gradient norm, applies AdamW
to each rank's fp32 master/m/v shard, casts to 16 bits and all-gathers the
result (ZeRO-1/2) or gathers per unit into a transient buffer (ZeRO-3).

The compute lives in ``libzero.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/zero.h``); :mod:`.binding` is a ctypes layer with the same
entry-point names.  The library is loaded on first use, not at import.
"""

__all__ = ["binding", "workloads", "synth"]
