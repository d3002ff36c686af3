"""CPU oracle for the DARTree draft-tree build and verify step.

TEST INFRASTRUCTURE ONLY. This is a plain, slow, float64 restatement of the
method for checking the CUDA path. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never calls it.

Sources (DARTree: Speculative Diffusion Decoding with Autoregressive Draft Trees,
as described on the marsggbo.github.io blog post "DARTree: ..."; section numbers
are that post's):
  * "3.1 Basic flow", candidate generation: keep the top-K tokens of each block
    position's base logits (default K = 64).
  * "3.1 Basic flow", depth-wise expansion: at depth d, all surviving parents of
    depth d-1 go through the correction head together, in one matrix operation.
  * "3.1 Basic flow", scoring function: s_beta(u_1:d) = sum_{i<=d} log q_i(u_i) + beta*d,
    beta <= 0.
  * "3.1 Basic flow", per-depth pruning: every depth keeps its top-W nodes.
  * "3.1 Basic flow", deferred pruning and Lemma 1: one global top-B over the
    supertree; for beta <= 0 this equals heap best-first popping.
  * "3.2": verification feeds all draft tokens to the target with a
    tree-attention mask and keeps the longest valid prefix.
  * ainews.surl.tw, "DARTree Builds Trees in Batches Before Pruning": same steps,
    16-token blocks, top-64 per position, depth reward non-positive.

The pages do not define the correction head. The stand-in head used here:
  u_p          = W_q h_p
  z[p, c]      = L^base[d-1, c] + <u_p, E[c]> / sqrt(H)
  q(c | p)     = softmax over the K candidates of position d-1
  h_child      = RMSNorm(h_p + E[tok] + H_d[d-1]), eps 1e-6, unit weight,
                 stored in the configuration's storage type (bf16 or fp32)
  h_root       = E[anchor], score 0, depth 0
Readings where the pages are silent (each is stated where it is used):
  * block row d-1 (0-based) feeds depth d; maximum depth is L;
  * top-W is taken jointly over all P*K children of a depth;
  * ties: top-K by lower token id; top-W by lower flat index p*K + c (p = parent
    rank, c = candidate rank); top-B by shallower depth, then lower rank;
  * output order is depth-major, rank within a depth; slot 0 is the root;
  * per-position target rows: the slot at depth delta is checked with row delta;
    per-node target rows: slot j is checked with row j.
"""
from __future__ import annotations

import heapq
import math

import numpy as np

from dartree_inputs import to_f64

RMS_EPS = 1e-6
TIE_TOL = 1e-3


# --------------------------------------------------------------------------- elementary steps

def round_bf16(x):
    """Round float64 values to the nearest bf16 value (8 significant bits), ties to even.

    Written from the definition: x = m * 2**e with 0.5 <= |m| < 1; keep 8 bits of m.
    Normal bf16 range only (the head state never leaves it).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_state(x, dtype: str):
    """Storage rounding of the head state: bf16 -> round_bf16, f32 -> float32."""
    if dtype == "bf16":
        return round_bf16(x)
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def topk_candidates(row, K: int):
    """Top-K of one position's base logits ("3.1", candidate generation).

    Order: logit descending, then token id ascending. Returns (tokens, logits).
    """
    order = np.argsort(-np.asarray(row, dtype=np.float64), kind="stable")[:K]
    return order.astype(np.int64), np.asarray(row, dtype=np.float64)[order]


def logsumexp(z):
    m = np.max(z)
    return m + math.log(float(np.sum(np.exp(z - m))))


def rmsnorm(x, eps: float = RMS_EPS):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def child_logits(h_par, cand_logit, Ec, Wq):
    """Corrected logits z[p, c] of every parent p over the K candidates of one position.

    Ec[c] = E[cand_tok[c]]. One matrix operation per depth over all parents
    ("3.1", depth-wise expansion).
    """
    H = Wq.shape[0]
    U = h_par @ Wq.T                      # u_p = W_q h_p   (rows of U)
    return cand_logit[None, :] + (U @ Ec.T) / math.sqrt(H)


def log_q(z):
    """log q = z - logsumexp_K(z), per parent row."""
    return np.stack([row - logsumexp(row) for row in z])


def score_children(s_par, logq, beta):
    """s_beta of every child: parent score + log q + beta ("3.1", scoring function).

    Accumulating the parent's score makes s the sum of log q over the path plus
    beta times the depth.
    """
    return s_par[:, None] + logq + beta


def depth_key(score, flat):
    """Per-depth order: score descending, then lower flat index p*K + c."""
    return (-score, flat)


def select_top(keys_desc, n: int):
    """Indices of the n best entries; keys_desc is a list of tuples compared ascending."""
    order = sorted(range(len(keys_desc)), key=lambda i: keys_desc[i])
    return order[:n]


# --------------------------------------------------------------------------- follow mode

def _adopt(own, other, score_of, valid, tol, what, flags, mismatches):
    """Compare an alternative ordered selection with the oracle's own.

    The alternative is adopted (and recorded in `flags` with its largest gap) only
    when it is a list of distinct valid entries of the same length and, at every
    rank position where the two lists differ, the two scores are unequal but
    within `tol` of each other: a near-tie that float32 arithmetic may order the
    other way. An exact tie (equal float64 scores) is not a near-tie: the stated
    tie order decides it, so a different choice there is a mismatch, like any
    gap of `tol` or more, a repeated entry or an unknown one. On a mismatch the
    oracle keeps its own choice.
    """
    if other is None or list(other) == list(own):
        return list(own)
    other = list(other)
    ok = len(other) == len(own) and len(set(other)) == len(other) and all(valid(x) for x in other)
    gaps = []
    if ok:
        gaps = [abs(score_of(a) - score_of(b)) for a, b in zip(own, other) if a != b]
        ok = all(0.0 < g < tol for g in gaps)
    if ok:
        flags.append((what, max(gaps, default=0.0)))
        return other
    mismatches.append(what)
    return list(own)


# --------------------------------------------------------------------------- tree build

class _Rows:
    """Float64 view of a stored [V, H] table that converts only the rows asked for."""

    def __init__(self, stored, dtype):
        self.stored, self.dtype = stored, dtype

    def __getitem__(self, idx):
        return to_f64(self.stored[idx], self.dtype)


def build(inp: dict, follow=None, tie_tol: float = TIE_TOL) -> dict:
    """Build the verification tree for every request of `inp`.

    follow: optional dict with callables 'depth'(i, d) -> ordered list of flat
    indices p*K + c, and 'prune'(i) -> list of (depth, rank); used to continue past
    a near-tie selection made by another implementation (see _adopt).
    """
    cfg = inp["cfg"]
    dt = cfg.dtype
    n = len(inp["anchor"])
    C_L_K = (n, cfg.L, cfg.K)
    out = dict(
        cand_tok=np.zeros(C_L_K, np.int64), cand_logit=np.zeros(C_L_K),
        st_tok=np.full((n, cfg.L, cfg.W), -1, np.int64), st_par=np.full((n, cfg.L, cfg.W), -1, np.int64),
        st_s=np.zeros((n, cfg.L, cfg.W)), st_n=np.zeros((n, cfg.L), np.int64),
        tok=np.full((n, cfg.B + 1), -1, np.int64), par=np.full((n, cfg.B + 1), -1, np.int64),
        depth=np.full((n, cfg.B + 1), -1, np.int64), score=np.zeros((n, cfg.B + 1)),
        n_nodes=np.zeros(n, np.int64), rank=np.full((n, cfg.B + 1), -1, np.int64),
        children=[[None] * cfg.L for _ in range(n)], flags=[], mismatches=[],
    )
    E = _Rows(inp["E"], dt)
    Wq = to_f64(inp["Wq"], dt)
    for i in range(n):
        _build_one(inp, i, E, Wq, out, follow, tie_tol)
    m, pos = mask_pos(out["par"], out["depth"], out["n_nodes"])
    out["mask"], out["pos"] = m, pos
    return out


def _build_one(inp, i, E, Wq, out, follow, tol):
    cfg = inp["cfg"]
    dt = cfg.dtype
    base = to_f64(inp["base"][i], dt)
    hid = to_f64(inp["hidden"][i], dt)
    L, K, W = cfg.L, cfg.K, cfg.W
    for j in range(L):
        out["cand_tok"][i, j], out["cand_logit"][i, j] = topk_candidates(base[j], K)
    # root: h = E[anchor], s = 0
    h = E[int(inp["anchor"][i])][None, :].copy()
    s = np.zeros(1)
    nodes = []  # (s, depth, rank, par_rank)
    for d in range(1, L + 1):
        ct, cl = out["cand_tok"][i, d - 1], out["cand_logit"][i, d - 1]
        z = child_logits(h, cl, E[ct], Wq)
        sc = score_children(s, log_q(z), cfg.beta)
        P = sc.shape[0]
        flat = sc.reshape(-1)
        out["children"][i][d - 1] = sc
        n_keep = min(W, P * K)
        own = select_top([depth_key(flat[f], f) for f in range(P * K)], n_keep)
        if follow is not None:
            own = _adopt(own, follow["depth"](i, d), lambda f: flat[f],
                         lambda f: isinstance(f, (int, np.integer)) and 0 <= f < P * K, tol,
                         ("depth", i, d), out["flags"], out["mismatches"])
        kept_par = [f // K for f in own]
        kept_c = [f % K for f in own]
        tok = ct[kept_c]
        x = h[kept_par] + E[tok] + hid[d - 1][None, :]
        h = round_state(rmsnorm(x), dt)
        s = flat[own]
        out["st_n"][i, d - 1] = n_keep
        out["st_tok"][i, d - 1, :n_keep] = tok
        out["st_par"][i, d - 1, :n_keep] = kept_par
        out["st_s"][i, d - 1, :n_keep] = s
        for k in range(n_keep):
            nodes.append((float(s[k]), d, k, kept_par[k]))
    prune_into(out, i, nodes, cfg.B, inp["anchor"][i], follow, tol)


def prune_into(out, i, nodes, B, anchor, follow=None, tol=TIE_TOL):
    """Deferred pruning ("3.1", Lemma 1): global top-B by (s desc, depth asc, rank asc),
    emitted depth-major with parents remapped to slot ids."""
    by_id = {(d, k): (s, p) for (s, d, k, p) in nodes}
    n_keep = min(B, len(nodes))
    order = select_top([(-s, d, k) for (s, d, k, _) in nodes], n_keep)
    chosen = [(nodes[t][1], nodes[t][2]) for t in order]
    if follow is not None:
        other = follow["prune"](i)
        if other is not None:
            other = sorted(other, key=lambda dk: (-by_id[dk][0], dk[0], dk[1])) \
                if all(dk in by_id for dk in other) else list(other)
        n_flags = len(out["flags"])
        kept = _adopt(chosen, other, lambda dk: by_id[dk][0], lambda dk: dk in by_id, tol,
                      ("prune", i), out["flags"], out["mismatches"])
        # an adopted set must still be prefix-closed (Lemma 1): every chosen node's
        # parent is chosen; otherwise it is a mismatch and the oracle's own set stays
        ks = set(kept)
        if len(out["flags"]) > n_flags and any(d > 1 and (d - 1, by_id[(d, k)][1]) not in ks for d, k in kept):
            del out["flags"][n_flags:]
            out["mismatches"].append(("prune", i))
        else:
            chosen = kept
    chosen = sorted(chosen)                       # depth-major, rank within depth
    slot_of = {(0, 0): 0}
    out["tok"][i, 0], out["par"][i, 0], out["depth"][i, 0] = anchor, -1, 0
    out["score"][i, 0], out["rank"][i, 0] = 0.0, 0
    for j, (d, k) in enumerate(chosen, start=1):
        s, p = by_id[(d, k)]
        slot_of[(d, k)] = j
        out["tok"][i, j] = out["st_tok"][i, d - 1, k]
        out["par"][i, j] = slot_of[(d - 1, p)] if d > 1 else 0
        out["depth"][i, j], out["score"][i, j], out["rank"][i, j] = d, s, k
    out["n_nodes"][i] = 1 + n_keep


def mask_pos(par, depth, n_nodes):
    """Tree-attention mask (ancestor-or-self) and position ids (= depth) ("3.2")."""
    n, S = par.shape
    mask = np.zeros((n, S, S), np.uint8)
    pos = np.full((n, S), -1, np.int64)
    for i in range(n):
        for a in range(int(n_nodes[i])):
            pos[i, a] = depth[i, a]
            b = a
            while b >= 0:
                mask[i, a, b] = 1
                b = par[i, b]
    return mask, pos


# --------------------------------------------------------------------------- verification

def verify(tree: dict, target: np.ndarray, dtype: str, rows: str, L: int) -> dict:
    """Greedy longest accepted prefix ("3.2": keep the longest valid prefix).

    From the root, t = argmax of the current slot's target row (lowest id among
    equal maxima); move to the child carrying t while one exists. Per-position
    rows: slot at depth delta uses row delta (no row at depth L, bonus -1).
    Per-node rows: slot j uses row j.
    """
    n = len(tree["n_nodes"])
    acc = np.zeros(n, np.int64)
    path = np.full((n, L), -1, np.int64)
    bonus = np.full(n, -1, np.int64)
    for i in range(n):
        nn = int(tree["n_nodes"][i])
        cur = 0
        while True:
            d = int(tree["depth"][i, cur])
            if rows == "position":
                if d >= L:
                    break
                row = to_f64(target[i, d], dtype)
            else:
                row = to_f64(target[i, cur], dtype)
            t = int(np.argmax(row))
            nxt = [j for j in range(1, nn) if tree["par"][i, j] == cur and tree["tok"][i, j] == t]
            if not nxt:
                bonus[i] = t
                break
            cur = nxt[0]
            path[i, acc[i]] = cur
            acc[i] += 1
    return dict(accepted_len=acc, path=path, bonus=bonus)


# --------------------------------------------------------------------------- reference searches

def heap_best_first(out, i, B):
    """Best-first popping on the materialised supertree (the heap side of Lemma 1).

    Start from the root's children; pop the best by (s desc, depth asc, rank asc);
    push the popped node's children. Returns popped (depth, rank) in pop order.
    """
    st_s, st_par, st_n = out["st_s"][i], out["st_par"][i], out["st_n"][i]
    L = st_s.shape[0]

    def kids(d, parent_rank):
        if d > L:
            return []
        return [(-float(st_s[d - 1, k]), d, k) for k in range(int(st_n[d - 1]))
                if d == 1 or st_par[d - 1, k] == parent_rank]

    heap = kids(1, 0)
    heapq.heapify(heap)
    popped = []
    while heap and len(popped) < B:
        _, d, k = heapq.heappop(heap)
        popped.append((d, k))
        for c in kids(d + 1, k):
            heapq.heappush(heap, c)
    return popped


def _head_per_node(h, pos, cand_tok, cand_logit, E, Wq):
    """Corrected log-probabilities for ONE parent, written with scalar loops.

    A second, independent formulation of the stand-in head (DDTree-style per-node
    correction, "2."): u_i = sum_j W_q[i][j] h[j]; z_c = base_c + sum_i u_i E[c][i] / sqrt(H).
    """
    H = len(h)
    u = [math.fsum(float(Wq[a][b]) * float(h[b]) for b in range(H)) for a in range(H)]
    z = [float(cand_logit[c]) + math.fsum(u[a] * float(E[int(cand_tok[c])][a]) for a in range(H)) / math.sqrt(H)
         for c in range(len(cand_tok))]
    m = max(z)
    lse = m + math.log(math.fsum(math.exp(v - m) for v in z))
    return [v - lse for v in z]


def _state_per_node(h, e, hd, dtype):
    H = len(h)
    x = [float(h[a]) + float(e[a]) + float(hd[a]) for a in range(H)]
    r = math.sqrt(math.fsum(v * v for v in x) / H + RMS_EPS)
    return round_state(np.array([v / r for v in x]), dtype)


def full_tree_heap(inp, i, B):
    """Best-first search over the unpruned K-ary tree, evaluating the head per popped
    node (node-by-node heap -> correction, "2."). Returns token paths in pop order."""
    cfg = inp["cfg"]
    dt = cfg.dtype
    E = _Rows(inp["E"], dt)
    Wq = to_f64(inp["Wq"], dt)
    base = to_f64(inp["base"][i], dt)
    hid = to_f64(inp["hidden"][i], dt)
    cands = [topk_candidates(base[j], cfg.K) for j in range(cfg.L)]
    root_h = E[int(inp["anchor"][i])]

    def expand(h, s, d, path, heap, counter):
        if d > cfg.L:
            return
        ct, cl = cands[d - 1]
        lq = _head_per_node(h, d - 1, ct, cl, E, Wq)
        for c in range(cfg.K):
            sc = s + lq[c] + cfg.beta
            heapq.heappush(heap, (-sc, d, next(counter), c, path, h, sc))

    import itertools
    counter = itertools.count()
    heap = []
    expand(root_h, 0.0, 1, (), heap, counter)
    popped = []
    while heap and len(popped) < B:
        negs, d, _, c, path, h_par, sc = heapq.heappop(heap)
        tok = int(cands[d - 1][0][c])
        newpath = path + (tok,)
        popped.append((newpath, sc))
        h = _state_per_node(h_par, E[tok], hid[d - 1], dt)
        expand(h, sc, d + 1, newpath, heap, counter)
    return popped


def tree_paths(out, i):
    """Token path (root excluded) and score of every slot of the built tree."""
    paths = []
    for j in range(1, int(out["n_nodes"][i])):
        p, b = [], j
        while b > 0:
            p.append(int(out["tok"][i, b]))
            b = int(out["par"][i, b])
        paths.append((tuple(reversed(p)), float(out["score"][i, j])))
    return paths
