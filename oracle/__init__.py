"""CPU oracle for the MoE layer hot path -- test infrastructure, not product code.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library and the
library never calls it.

Parity status per function (what pins each one to something other than itself
is listed in tests/test_oracle_pins.py):
  route_softmax, route_sigmoid_group, sigmoid_det_f32, permute, combine,
  pool_pack, pool_compact, compose_map, capacity helpers: pinned.
  swiglu / grouped_swiglu_rows: pinned by special cases only (dense reduction
  against an independent matmul, fused-equals-sum, closed form at d=I=1, and
  several segments with distinct scalar experts, each row against its own
  expert's closed form); the pages print no SwiGLU output values.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import EMPTY_HEADER  # noqa: F401
