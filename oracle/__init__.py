"""fp64 CPU oracle of the routed-expert MoE layer (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may use it.  The library's CUDA path does not import it and shares no code
with it.  See ``moe_oracle.py`` for the steps and the passages they follow.
"""
from .moe_oracle import (  # noqa: F401
    as_f64,
    decode_bf16,
    dequant_affine4,
    group,
    moe_layer,
    route,
    router_logits,
    select_top_k,
    sigmoid,
    silu,
    softmax,
    swiglu_ffn,
    unpack_u4,
)
