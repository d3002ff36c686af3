"""CPU oracle of the DARTree draft-tree build and verify step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
package; the library and its Python binding never do.
"""
from .dartree import (  # noqa: F401
    RMS_EPS, TIE_TOL, build, child_logits, full_tree_heap, heap_best_first, log_q,
    logsumexp, mask_pos, prune_into, rmsnorm, round_bf16, round_state, topk_candidates,
    tree_paths, verify,
)
from . import sampling  # noqa: F401,E402  (temperature-T verification, adaptive budget)
from . import lm_head  # noqa: F401,E402  (stand-in LM head followed by S1)
from . import tree_attention  # noqa: F401,E402  (the verification pass's tree attention)
