"""CPU oracle for the W4 group-affine sparse-MoE layer.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and by
the benchmark's CPU-baseline leg, never by the CUDA library or its binding.

Pinned functions (each checked by tests/test_oracle_pins.py against values
fixed by the pages or by mathematics, not against itself):
  unpack_codes, dequant, e4m3_value, bits_per_weight, route (select_top_k,
  softmax renormalisation, shared gate), group, block_map, silu, expert_ffn,
  moe_layer.
No function is "parity unpinned".
"""
from .moe_w4_oracle import *  # noqa: F401,F403
from .moe_w4_oracle import (bf16_to_f64, f64_to_bf16, unpack_codes, dequant, route, group,  # noqa: F401
                            block_map, silu, expert_ffn, moe_layer, select_top_k, router_scores,
                            bits_per_weight, checkpoint_gb, sigmoid, e4m3_value, CODES_UINT, CODES_E4M3)
