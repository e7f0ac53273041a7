"""GB300-native MoE layer hot path: route -> permute -> grouped SwiGLU GEMM -> combine,
plus the static-shape pooled-wave layout, as hand-written sm_103a CUDA behind a C ABI
(include/moe.h).  ``abi`` is the thin ctypes binding with the C names; ``layer``
composes the calls into one layer forward.
"""
from . import abi  # noqa: F401
from .abi import *  # noqa: F401,F403
from .layer import (DecodeBucket, DecodeBucketLadder, HostPipeline, MoELayer,  # noqa: F401
                    PooledMoELayer, capacity_from_factor)

__all__ = ["abi", "MoELayer", "PooledMoELayer", "DecodeBucket", "DecodeBucketLadder", "HostPipeline",
           "capacity_from_factor"] + abi.EXPORTED
