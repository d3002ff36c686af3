"""CPU oracle of verification at a temperature T > 0, and of the adaptive budget policy.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it.

The pages report DARTree at temperatures 0 and 1 and call the speed-up lossless
(DARTree blog post, section 4 and Table 1; ainews.surl.tw, "DARTree Builds Trees in
Batches Before Pruning", evaluation paragraph), but print no acceptance rule for
T > 0. The rule restated here is the plainest lossless one for a tree whose children
are chosen deterministically (top-K, top-W, top-B, not sampled from the draft):

  * at every step the target's token is DRAWN from softmax(row / T) of the current
    slot's target row, by the Gumbel-max construction:
        t = argmax_v ( x_v / T + G_v ),   G_v = -log(-log U_v),   U_v ~ U(0, 1);
    equal perturbed values go to the lower token id;
  * the walk moves to the child carrying t while one exists, else t is the bonus
    token and the walk ends (the same walk as greedy verification, "3.2").
Every emitted token (accepted drafts and the bonus) is therefore an exact sample of
the target at temperature T given the tokens before it, whatever the tree holds: the
output distribution is the target's own (lossless). As T -> 0 it becomes the greedy
rule of verify().

Random numbers: U_v comes from one counter-based generator, Philox4x32-10 (J. Salmon,
M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011),
written out below from that definition:
  key     (seed mod 2^32, seed div 2^32)
  counter (v div 4, row, request, 0), output word v mod 4
  U       (2 * (word >> 9) + 1) * 2^-24         (exact in float32, inside (0, 1))
where row is the depth delta of the slot for per-position target rows and the slot
index j for per-node rows. The decision is taken in float32 (x_v / T and the sum
rounded to float32, the logarithms in float32), the precision of the kernel.

Adaptive budget (blog section 4.4): at concurrency C = 4 the pages shrink the node
budget B from 64 to 32 and the width W from 12 to 3; at C = 1 and C = 2 they run the
defaults. Reading: the reduced budget applies from C = 4 on (the smallest
concurrency the pages use it at); below C = 4 the defaults hold.
"""
from __future__ import annotations

import numpy as np

from dartree_inputs import to_f32

MASK32 = 0xFFFFFFFF
# Philox4x32 multipliers and Weyl key increments (Salmon et al. 2011)
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
PHILOX_ROUNDS = 10

DEFAULT_BUDGET = (64, 12)   # (B, W) at C < 4
REDUCED_BUDGET = (32, 3)    # (B, W) at C >= 4
REDUCED_FROM_C = 4


def philox4x32(ctr, key, rounds: int = PHILOX_ROUNDS):
    """Philox4x32-R on 32-bit words held in numpy uint64 arrays (broadcast together).

    One round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products), then
    c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key gains the Weyl
    increments (W0, W1) before every round but the first.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & np.uint64(MASK32) for c in ctr)
    k0, k1 = int(key[0]) & MASK32, int(key[1]) & MASK32
    m0, m1, mask = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1), np.uint64(MASK32)
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + PHILOX_W0) & MASK32, (k1 + PHILOX_W1) & MASK32
        p0 = m0 * c0
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0
    return c0, c1, c2, c3


def uniforms(seed: int, request: int, row: int, V: int) -> np.ndarray:
    """U_v for v = 0..V-1 of one (request, row), float32, inside (0, 1)."""
    v = np.arange(V, dtype=np.uint64)
    words = philox4x32((v >> np.uint64(2), np.uint64(row), np.uint64(request), np.uint64(0)),
                       (seed & MASK32, (seed >> 32) & MASK32))
    w = np.choose((v & np.uint64(3)).astype(np.int64), words)
    num = (w >> np.uint64(9)) * np.uint64(2) + np.uint64(1)   # odd, < 2^24: exact in float32
    return num.astype(np.float32) * np.float32(2.0 ** -24)


def perturbed(row_f32: np.ndarray, T: float, U: np.ndarray) -> np.ndarray:
    """x_v / T + G_v in float32, G_v = -log(-log U_v)."""
    g = -np.log(-np.log(U.astype(np.float32)))
    return (row_f32.astype(np.float32) / np.float32(T) + g.astype(np.float32)).astype(np.float32)


def sample_token(row_f32: np.ndarray, T: float, seed: int, request: int, row: int):
    """Gumbel-max draw from softmax(row / T): (token, margin), margin = the gap to the
    runner-up's perturbed value (how close the decision was)."""
    y = perturbed(row_f32, T, uniforms(seed, request, row, row_f32.shape[0]))
    t = int(np.argmax(y))  # first maximum: the lowest token id among equal values
    if y.shape[0] < 2:
        return t, float("inf")
    rest = np.delete(y, t)
    return t, float(y[t]) - float(rest.max())


def verify_sample(tree: dict, target: np.ndarray, dtype: str, rows: str, L: int, T: float, seed: int,
                  requests=None) -> dict:
    """Longest accepted prefix when the target samples at temperature T (rule above).

    Same walk and outputs as verify(); per-position rows: the slot at depth delta uses
    row delta (no row at depth L: bonus -1); per-node rows: slot j uses row j. Also
    returns the smallest decision margin met on the walks. requests: the request
    index of each entry in the counter (default 0, 1, ...), so that a sample of a
    batch can be checked on its own.
    """
    if not (T > 0 and np.isfinite(T)):
        raise ValueError("temperature must be positive and finite")
    n = len(tree["n_nodes"])
    req = np.arange(n) if requests is None else np.asarray(requests)
    acc = np.zeros(n, np.int64)
    path = np.full((n, L), -1, np.int64)
    bonus = np.full(n, -1, np.int64)
    min_margin = float("inf")
    for i in range(n):
        nn = int(tree["n_nodes"][i])
        cur = 0
        while True:
            d = int(tree["depth"][i, cur])
            if rows == "position":
                if d >= L:
                    break
                rid, row = d, to_f32(target[i, d], dtype)
            else:
                rid, row = cur, to_f32(target[i, cur], dtype)
            t, margin = sample_token(row, T, seed, int(req[i]), rid)
            min_margin = min(min_margin, margin)
            nxt = [j for j in range(1, nn) if tree["par"][i, j] == cur and tree["tok"][i, j] == t]
            if not nxt:
                bonus[i] = t
                break
            cur = nxt[0]
            path[i, acc[i]] = cur
            acc[i] += 1
    return dict(accepted_len=acc, path=path, bonus=bonus, min_margin=min_margin)


def adaptive_budget(C: int) -> tuple[int, int]:
    """(B, W) for concurrency C (blog section 4.4; reading in the module docstring)."""
    if C < 1:
        raise ValueError("concurrency must be at least 1")
    return REDUCED_BUDGET if C >= REDUCED_FROM_C else DEFAULT_BUDGET
