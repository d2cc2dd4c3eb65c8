"""Routed-expert W4A8 MoE layer for GB300 (sm_103a).

The layer routes each token to its top-k experts on the device, groups the
(token, expert) pairs per expert with a stable counting sort, and runs the
grouped gate/up and down projections directly on a packed int4 expert bank
with per-group fp32 scales and per-token int8 activations, followed by
SiLU(gate) * up, a per-row int8 requantisation and a routing-weighted
combine.  All of it runs in the CUDA kernels of ``libmoe_w4a8.so``; this
package only marshals arguments to its C ABI (``include/moe_w4a8.h``).

Attributes of the binding (``moe_w4a8_forward`` and friends) load the
library on first use and raise if it is missing; nothing falls back to a
CPU implementation.
"""
from __future__ import annotations

__all__ = ["moe_w4a8_forward", "moe_w4a8_route", "moe_w4a8_gemm1_partials", "moe_w4a8_gemm2_partials",
           "moe_w4a8_workspace_size", "moe_w4a8_version", "moe_w4a8_status_string", "moe_w4a8_forward_noalloc",
           "Dims", "MoeError"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
