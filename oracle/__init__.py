"""fp64 CPU oracle (test infrastructure only; see ``oracle.attention``)."""
from .attention import (NEG_INF, allowed_mask, allowed_rows, attention_backward,
                        attention_forward, backward_head, blocklist_normalize,
                        blocklist_stats,
                        blocklist_sets, executed_tiles, finalize_state, forward_head,
                        kv_group, logical_pairs, merge_pair, merge_states, partial_state,
                        probabilities)

__all__ = [
    "NEG_INF", "allowed_mask", "allowed_rows", "attention_backward", "attention_forward",
    "backward_head", "blocklist_normalize", "blocklist_sets", "blocklist_stats", "executed_tiles",
    "finalize_state", "forward_head", "kv_group", "logical_pairs", "merge_pair", "merge_states",
    "partial_state", "probabilities",
]
