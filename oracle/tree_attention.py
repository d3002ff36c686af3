"""CPU oracle of the verification pass's tree attention over a KV cache.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it.

DARTree hands the pruned tree to the target model, which checks every drafted
token in one forward pass with a tree-attention mask (DARTree blog post, "3.2";
ainews.surl.tw, "DARTree Builds Trees in Batches Before Pruning": one tree-attention
operation). The pages do not print the attention; the plain reading used here is
one causal-attention layer of the target in which the tree tokens attend to
  * every cached token of the request's prefix (positions 0 .. n_ctx - 1), and
  * the tree slots the mask marks visible (ancestor-or-self, from S9),
with rotary position embedding at position n_ctx + pos[j] for tree slot j (pos =
the slot's depth, from S9; the root sits at n_ctx). Conventions of the Qwen3 target
models the pages evaluate: grouped-query attention (query head h reads key/value
head h // (Hq / Hkv)), scores scaled by 1 / sqrt(D), rotary pairs (i, i + D/2) with
inverse frequency theta^(-2i / D). The cached keys are stored already rotated; the
tree's queries and keys arrive unrotated (after the projections and their norms,
which are not part of this step). Unused slots (j >= n_nodes) give zero rows.

Everything is computed in float64 from the stored values.
"""
from __future__ import annotations

import numpy as np

from dartree_inputs import to_f64

ROPE_THETA = 1.0e6


def rope(x: np.ndarray, positions: np.ndarray, theta: float = ROPE_THETA) -> np.ndarray:
    """Rotate the last axis (D, even) of x [..., n, D] by position positions[n]:
    x'_i = x_i cos(a_i) - x_{i+D/2} sin(a_i), x'_{i+D/2} = x_{i+D/2} cos(a_i) + x_i sin(a_i),
    a_i = p * theta^(-2i/D), i < D/2."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    ang = np.asarray(positions, np.float64)[:, None] * inv[None, :]       # [n, D/2]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def tree_attention(q, k_tree, v_tree, k_cache, v_cache, n_ctx, mask, pos, n_nodes, dtype: str,
                   theta: float = ROPE_THETA):
    """Output [C, S, Hq, D] (float64) of one tree-attention layer.

      q        [C, S, Hq, D]    tree queries (unrotated), stored values
      k_tree   [C, S, Hkv, D]   tree keys (unrotated)
      v_tree   [C, S, Hkv, D]   tree values
      k_cache  [C, Hkv, N, D]   prefix keys (rotated), positions 0..N-1
      v_cache  [C, Hkv, N, D]   prefix values
      n_ctx    [C]              cached prefix length of each request (<= N)
      mask     [C, S, S]        1 where slot j sees slot i (S9)
      pos      [C, S]           slot depths (S9), -1 for unused slots
      n_nodes  [C]              used slots
    """
    C, S, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    grp = Hq // Hkv
    out = np.zeros((C, S, Hq, D), np.float64)
    for c in range(C):
        n = int(n_nodes[c])
        nc = int(n_ctx[c])
        p = nc + np.asarray(pos[c, :n], np.int64)
        qr = rope(np.moveaxis(to_f64(q[c, :n], dtype), 0, 1), p, theta)          # [Hq, n, D]
        kr = rope(np.moveaxis(to_f64(k_tree[c, :n], dtype), 0, 1), p, theta)     # [Hkv, n, D]
        vt = np.moveaxis(to_f64(v_tree[c, :n], dtype), 0, 1)                     # [Hkv, n, D]
        kc = to_f64(k_cache[c, :, :nc], dtype)                                   # [Hkv, nc, D]
        vc = to_f64(v_cache[c, :, :nc], dtype)
        for h in range(Hq):
            g = h // grp
            keys = np.concatenate([kc[g], kr[g]], axis=0)
            vals = np.concatenate([vc[g], vt[g]], axis=0)
            for j in range(n):
                seen = np.concatenate([np.ones(nc, bool), np.asarray(mask[c, j, :n], bool)])
                s = keys[seen] @ qr[h, j] / np.sqrt(D)
                w = np.exp(s - s.max())
                out[c, j, h] = (w / w.sum()) @ vals[seen]
    return out
