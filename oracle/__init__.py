"""CPU oracle for the MegaMoE forward (test infrastructure only; see moe_oracle)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (E4M3, E2M1, bf16_rne, dequant_weight, dequant_x, e2m1_decode,  # noqa: F401
                         e4m3_decode, e4m3_encode_rne, expert_from_arrays, forward, forward_pair,
                         requant_f8, requant_mx, route, ue8m0_decode, ue8m0_exponent)
