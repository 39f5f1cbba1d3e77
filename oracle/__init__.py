"""Oracle of the dropless MoE layer forward -- TEST INFRASTRUCTURE.

A plain, slow CPU implementation (fp32 router logits with a fixed rounding
order, fp64 for everything after them) that the CUDA library is checked
against.  Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs use it; the library never imports it.
"""
from .moe_oracle import (combine, dispatch_order, expert_counts, expert_ffn, forward,  # noqa: F401
                         forward_tokens, grouped_mlp, host_threads, permute, router_logits_fp32,
                         router_logits_fp64, silu, topk_route)
from .mxfp8 import (e4m3_decode, e4m3_encode, e4m3_round, expert_ffn_mxfp8, forward_mxfp8,  # noqa: F401
                    forward_mxfp8_tokens, mx_dequantize, mx_quantize, mx_scale_exponent)
from .backward import backward, backward_sampled, forward_fp64  # noqa: F401
