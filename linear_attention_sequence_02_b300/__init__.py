"""B300-native RetNet multi-scale retention.

The compute lives in ``libretention.so`` (hand-written sm_103a CUDA behind a
plain C ABI, declared in ``include/retention.h``).  This package holds the
thin ctypes binding (:mod:`.binding`), the build step (:mod:`.build`) and the
seeded input generators (:mod:`.inputs`).  The binding loads the library on
first use and raises if it is missing; there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    RetentionError,
    gamma_schedule,
    retention_chunkwise,
    retention_chunkwise_f32,
    retention_parallel,
    retention_parallel_f32,
    retention_step,
    retention_step_f32,
)

__all__ = [
    "RetentionError",
    "gamma_schedule",
    "retention_chunkwise",
    "retention_chunkwise_f32",
    "retention_parallel",
    "retention_parallel_f32",
    "retention_step",
    "retention_step_f32",
]
