"""fp64 CPU oracle for exact shared-prompt attention (test infrastructure only;
the product path never imports it)."""
from .attention import (causal_attention_bwd, causal_attention_fwd, dualkv_backward,
                        dualkv_forward, keys_dkdv, rows_forward_backward, segment_offsets)

__all__ = ["causal_attention_fwd", "causal_attention_bwd", "dualkv_forward", "dualkv_backward",
           "rows_forward_backward", "keys_dkdv", "segment_offsets"]
