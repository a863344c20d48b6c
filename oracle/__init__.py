"""CPU oracle (test infrastructure only; see ``oracle.attention``)."""
from .attention import *  # noqa: F401,F403
from .attention import (attention, attention_rows, attention_bwd, attention_bwd_partial, merge, merge_pair,
                        ring_forward, usp_forward, allgather_forward, ring_positions, shard, unshard,
                        ulysses_seq_to_head, ulysses_head_to_seq, ulysses_lse_head_to_seq,
                        visible, doc_start_of, visible_pairs, rank_visible_pairs,
                        chunk_work, balanced_chunks,
                        LAYOUT_CONTIGUOUS, LAYOUT_ZIGZAG, LAYOUT_BALANCED)  # noqa: F401
