"""libbeamnorm: the arithmetic epilogue of a fused tensor-parallel all-reduce
(rank-ordered FP32 sum of R BF16 shards, optional per-shard MoE top-k
finalize, post-RMSNorm, residual add, next-layer RMSNorm) on one GB300.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/beamnorm.h``); ``beamnorm`` is the Python binding and ``inputs``
draws the seeded synthetic workloads.
"""
from .beamnorm import (BeamNormError, Debug, check_device_error, finalize_only,  # noqa: F401
                       finalize_reduce_norm, finalize_reduce_only,
                       finalize_reduce_residual_norm, norm_only, reduce_norm, reduce_only,
                       reduce_residual_norm, set_tuning, supports, version)
