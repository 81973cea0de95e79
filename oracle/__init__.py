"""Float64 CPU oracle of the token-selection path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product path never does.
"""
from .upf_oracle import (bf16_to_f64, tail_positions, kv_head_map, token_scores, block_means,  # noqa: F401
                         top_p_blocks, exempt_blocks, select, compact, select_tokens, history_kv_len, revive)
