"""Float64 CPU oracle of the dropless MoE expert layer.

Test infrastructure only: used by tests/, __graft_entry__.smoke() and the CPU
baseline legs of bench.py; the CUDA library never imports it."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (route, route_backward, permute, forward, backward,  # noqa: F401
                         quantize_mxfp8, dequantize_mxfp8, e4m3_round,
                         e4m3_encode, e4m3_decode, mx_block_exponent, mx_qdq,
                         rel_err, bf16_round, ALIGN, MX_BLOCK)
