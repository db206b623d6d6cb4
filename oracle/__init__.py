"""CPU oracle for masked attention: TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 restatement of what the attention path computes, used to
check the CUDA library. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the library itself never does.
Every function is pinned by ``tests/test_oracle.py`` against closed forms,
invariants, brute force and a library special case.
"""
from .attention import (Spec, alibi_slopes, mask_mod, score_mod, score_mod_grad,
                        attention_forward, attention_backward, block_mask, BlockMask,
                        kept_per_row, combine_partials)

__all__ = ["Spec", "alibi_slopes", "mask_mod", "score_mod", "score_mod_grad",
           "attention_forward", "attention_backward", "block_mask", "BlockMask",
           "kept_per_row", "combine_partials"]
