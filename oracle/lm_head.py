"""CPU oracle of the block drafter's LM head followed by S1 (candidate generation).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it.

DARTree keeps the top-K tokens of every block position's base logits (DARTree blog
post, "3.1 Basic flow", candidate generation; ainews.surl.tw, "DARTree Builds Trees
in Batches Before Pruning": top-64 per position). The base logits are the block
drafter's LM head applied to its hidden states; the pages do not print the head, so
the stand-in is a plain linear map without bias:
    L^base[r, v] = <h_r, W_lm[v]>,   h_r = H_d row r (one row per request and position),
and S1 keeps, per row, the K largest logits, ordered by logit descending, then
token id ascending (the same tie rule as S1 on stored logits).

The logits here are the exact dot products of the stored (bf16 or fp32) values,
summed in float64; a fused kernel that never writes them may differ from them by its
own accumulation rounding only.
"""
from __future__ import annotations

import numpy as np

from dartree_inputs import to_f64

from .dartree import topk_candidates

CHUNK_ROWS = 8192   # vocabulary rows converted to float64 at a time


def lm_head_logits(hidden: np.ndarray, W_lm: np.ndarray, dtype: str) -> np.ndarray:
    """Base logits [R, V] in float64: hidden [R, H] against every vocabulary row of W_lm [V, H]."""
    h = to_f64(np.asarray(hidden), dtype)
    V = W_lm.shape[0]
    out = np.empty((h.shape[0], V), np.float64)
    for v0 in range(0, V, CHUNK_ROWS):
        v1 = min(V, v0 + CHUNK_ROWS)
        out[:, v0:v1] = h @ to_f64(W_lm[v0:v1], dtype).T
    return out


def lm_head_topk(hidden: np.ndarray, W_lm: np.ndarray, K: int, dtype: str):
    """S1 on the LM head's logits: (tok [R, K], logit [R, K], logits [R, V])."""
    logits = lm_head_logits(hidden, W_lm, dtype)
    R = logits.shape[0]
    tok = np.empty((R, K), np.int64)
    val = np.empty((R, K), np.float64)
    for r in range(R):
        tok[r], val[r] = topk_candidates(logits[r], K)
    return tok, val, logits
