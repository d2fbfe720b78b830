"""fp64 CPU oracle (test infrastructure only; see fp64.py)."""
from .fp64 import (default_sections, token_positions, rope_frequencies,  # noqa: F401
                               rope3d_angles, apply_rotary, rope3d, attention_rows,
                               rope3d_attention, rope3d_attention_rows,
                   block_key_mask, attention_rows_masked, rope3d_attention_blocksparse,
                   window_block_mask, rope3d_attention_blocksparse_rows)
