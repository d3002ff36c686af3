"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the method (DARTree blog post, sections 2, 3.1 and 3.2)
by a worked example derived by hand, a library routine, a closed form, a special
case the pages name, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import dartree as od
from dartree_inputs import bf16_bits_to_f32, round_to_bf16_bits, to_f64
from _tiny import golden_inputs, load_golden, tiny_inputs

G = load_golden("closed_form_tree.json")


def _closed_form_scores(dtype):
    env = dict(log=math.log, exp=math.exp, sqrt=math.sqrt, beta=G["config"]["beta"])
    env["a"] = eval(G["expected"]["a"][dtype], {}, env)
    sc = G["expected"]["scores"]
    for k in ("s1_0", "s1_1", "f1", "f2"):
        env[k] = eval(sc[k], {}, env)
    return env


# --------------------------------------------------------------------------- worked example

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_closed_form_worked_example(dtype):
    inp = golden_inputs(G, dtype)
    out = oracle.build(inp)
    ex = G["expected"]
    for k in ("cand_tok", "st_tok", "st_par", "tok", "par", "depth", "n_nodes", "mask", "pos"):
        np.testing.assert_array_equal(out[k], np.asarray(ex[k]), err_msg=k)
    env = _closed_form_scores(dtype)
    np.testing.assert_allclose(out["st_s"][0], [[env["s1_0"], env["s1_1"]], [env["f1"], env["f2"]]],
                               rtol=0, atol=1e-6)
    np.testing.assert_allclose(out["score"][0], [0, env["s1_0"], env["s1_1"], env["f1"]], rtol=0, atol=1e-6)
    v = oracle.verify(out, inp["target"], dtype, "position", inp["cfg"].L)
    assert v["accepted_len"].tolist() == ex["accepted_len"]
    assert v["path"].tolist() == ex["path"]
    assert v["bonus"].tolist() == ex["bonus"]


# --------------------------------------------------------------------------- elementary steps

def test_round_bf16_matches_bit_level_rounding():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10,
                        rng.standard_normal(2000).astype(np.float32) * 1e-3])
    ref = bf16_bits_to_f32(round_to_bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(od.round_bf16(x.astype(np.float64)), ref)
    # ties to even, exactly half way between two bf16 values
    assert od.round_bf16(1 + 2**-8) == 1.0
    assert od.round_bf16(1 + 3 * 2**-8) == 1 + 2**-6
    assert od.round_bf16(-(1 + 3 * 2**-8)) == -(1 + 2**-6)
    assert od.round_bf16(math.sqrt(2)) == 1.4140625


def test_topk_against_bruteforce_with_ties():
    rng = np.random.default_rng(3)
    for _ in range(50):
        V = int(rng.integers(2, 60))
        row = rng.integers(-3, 4, size=V).astype(np.float64)
        K = int(rng.integers(1, V + 1))
        tok, val = od.topk_candidates(row, K)
        ref = sorted(range(V), key=lambda t: (-row[t], t))[:K]
        assert tok.tolist() == ref
        assert val.tolist() == [row[t] for t in ref]


def test_logsumexp_and_softmax_normalisation():
    rng = np.random.default_rng(5)
    for _ in range(20):
        z = rng.standard_normal(37) * 20
        assert abs(od.logsumexp(z) - scipy.special.logsumexp(z)) < 1e-12
        q = np.exp(od.log_q(z[None, :])[0])
        assert abs(q.sum() - 1.0) < 1e-12


def test_rmsnorm_closed_form():
    x = np.array([1.0, 0.0, 1.0, 0.0])
    np.testing.assert_allclose(od.rmsnorm(x), x / math.sqrt(0.5 + 1e-6), rtol=1e-15)
    y = np.array([3.0, -4.0])
    np.testing.assert_allclose(od.rmsnorm(y), y / math.sqrt(12.5 + 1e-6), rtol=1e-15)


# --------------------------------------------------------------------------- Lemma 1 and the named special cases

SEEDS = range(12)


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("ties", [False, True])
def test_lemma1_global_topB_equals_heap_best_first(seed, ties):
    """Lemma 1 ("3.1", deferred pruning): for beta <= 0 the global top-B of the
    supertree equals best-first heap popping on it, and is prefix-closed."""
    rng = np.random.default_rng(seed)
    beta = float(-rng.uniform(0, 1)) if seed % 3 else 0.0
    inp = tiny_inputs(seed, ties=ties, L=int(rng.integers(1, 5)), K=int(rng.integers(1, 4)),
                      W=int(rng.integers(1, 4)), B=int(rng.integers(1, 9)), beta=beta)
    out = oracle.build(inp)
    n_sel = int(out["n_nodes"][0]) - 1
    chosen = sorted((int(out["depth"][0, j]), int(out["rank"][0, j])) for j in range(1, n_sel + 1))
    popped = od.heap_best_first(out, 0, inp["cfg"].B)
    assert sorted(popped) == chosen
    # prefix closure: every chosen node's parent is the root or a chosen node
    for j in range(1, n_sel + 1):
        p = int(out["par"][0, j])
        assert p == 0 or (0 < p < j and out["depth"][0, p] == out["depth"][0, j] - 1)


@pytest.mark.parametrize("seed", SEEDS)
def test_scores_never_increase_along_a_path(seed):
    """beta <= 0 and log q <= 0 make s_child <= s_parent (the invariant behind Lemma 1)."""
    inp = tiny_inputs(seed, beta=-0.05 * (seed % 4))
    out = oracle.build(inp)
    for j in range(1, int(out["n_nodes"][0])):
        p = int(out["par"][0, j])
        assert out["score"][0, j] <= out["score"][0, p]


@pytest.mark.parametrize("seed", SEEDS)
def test_w1_gives_a_single_chain(seed):
    """W = 1 keeps one node per depth: a Domino-style chain ("2.")."""
    inp = tiny_inputs(seed, L=5, K=4, W=1, B=8)
    out = oracle.build(inp)
    L = inp["cfg"].L
    assert out["n_nodes"][0] == 1 + L
    assert out["par"][0, 1:L + 1].tolist() == list(range(L))
    for d in range(1, L + 1):
        ch = out["children"][0][d - 1]
        assert ch.shape[0] == 1
        c = int(np.argmax(ch[0]))
        assert out["st_tok"][0, d - 1, 0] == out["cand_tok"][0, d - 1, c]
    m = out["mask"][0, :L + 1, :L + 1]
    np.testing.assert_array_equal(m, np.tril(np.ones((L + 1, L + 1), np.uint8)))


@pytest.mark.parametrize("seed", SEEDS)
def test_k1_gives_the_base_argmax_chain(seed):
    """K = 1: every node is its position's base argmax, q = 1 and s = beta*d (DFlash chain)."""
    inp = tiny_inputs(seed, L=6, K=1, W=3, B=10, beta=-0.25)
    out = oracle.build(inp)
    base = to_f64(inp["base"][0], "f32")
    L = inp["cfg"].L
    assert out["n_nodes"][0] == 1 + L
    for d in range(1, L + 1):
        assert out["tok"][0, d] == int(np.argmax(base[d - 1]))
        assert out["score"][0, d] == -0.25 * d


@pytest.mark.parametrize("seed", SEEDS)
def test_beta0_orders_by_cumulative_log_probability(seed):
    """beta = 0: every supertree node's score is its path's sum of log q, here
    recomputed node by node with the scalar head; the top-B set is the best B of those."""
    inp = tiny_inputs(seed, L=3, K=3, W=3, B=5, beta=0.0)
    out = oracle.build(inp)
    cfg = inp["cfg"]
    E = to_f64(inp["E"], "f32")
    Wq = to_f64(inp["Wq"], "f32")
    hid = to_f64(inp["hidden"][0], "f32")
    cum = {}
    states = {(0, 0): E[int(inp["anchor"][0])]}
    for d in range(1, cfg.L + 1):
        for k in range(int(out["st_n"][0, d - 1])):
            p = int(out["st_par"][0, d - 1, k])
            tok = int(out["st_tok"][0, d - 1, k])
            ct, cl = out["cand_tok"][0, d - 1], out["cand_logit"][0, d - 1]
            lq = od._head_per_node(states[(d - 1, p)], d - 1, ct, cl, E, Wq)
            c = int(np.where(ct == tok)[0][0])
            cum[(d, k)] = cum.get((d - 1, p), 0.0) + lq[c]
            states[(d, k)] = od._state_per_node(states[(d - 1, p)], E[tok], hid[d - 1], "f32")
            assert abs(cum[(d, k)] - out["st_s"][0, d - 1, k]) < 1e-9
    best = sorted(cum, key=lambda dk: (-cum[dk], dk))[:cfg.B]
    chosen = sorted((int(out["depth"][0, j]), int(out["rank"][0, j])) for j in range(1, int(out["n_nodes"][0])))
    assert sorted(best) == chosen


@pytest.mark.parametrize("seed", SEEDS)
def test_w_at_least_b_equals_node_by_node_heap_on_the_full_tree(seed):
    """W >= B: the deferred tree equals best-first search on the unpruned K-ary tree
    with the head evaluated per popped node (DDTree-style heap -> correction, "2.")."""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 7))
    inp = tiny_inputs(seed, L=4, K=3, W=B + int(rng.integers(0, 2)), B=B, beta=-float(rng.uniform(0, 0.5)))
    out = oracle.build(inp)
    ref = od.full_tree_heap(inp, 0, B)
    got = od.tree_paths(out, 0)
    assert sorted(p for p, _ in got) == sorted(p for p, _ in ref)
    ref_s = dict(ref)
    for p, s in got:
        assert abs(ref_s[p] - s) < 1e-9


@pytest.mark.parametrize("seed", SEEDS)
def test_supertree_does_not_depend_on_beta(seed):
    """beta*d is the same for all nodes of a depth, so per-depth top-W ignores beta."""
    a = oracle.build(tiny_inputs(seed, beta=0.0))
    b = oracle.build(tiny_inputs(seed, beta=-0.7))
    for k in ("st_tok", "st_par", "st_n"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("seed", SEEDS)
def test_very_negative_beta_fills_breadth_first(seed):
    inp = tiny_inputs(seed, L=4, K=3, W=3, B=7, beta=-1e6)
    out = oracle.build(inp)
    d = out["depth"][0, 1:int(out["n_nodes"][0])]
    full = [int(out["st_n"][0, i]) for i in range(4)]
    expect = []
    for depth, cnt in enumerate(full, start=1):
        expect += [depth] * cnt
    assert d.tolist() == expect[:7]


@pytest.mark.parametrize("seed", SEEDS)
def test_mask_invariants(seed):
    out = oracle.build(tiny_inputs(seed, L=4, K=3, W=3, B=8))
    n = int(out["n_nodes"][0])
    m = out["mask"][0]
    assert np.all(np.triu(m[:n, :n], 1) == 0)
    assert np.all(np.diag(m[:n, :n]) == 1)
    np.testing.assert_array_equal(m[:n, :n].sum(1), out["depth"][0, :n] + 1)
    for j in range(1, n):
        assert m[j, out["par"][0, j]] == 1
    assert np.all(m[n:] == 0) and np.all(m[:, n:] == 0)
    np.testing.assert_array_equal(out["pos"][0, :n], out["depth"][0, :n])


# --------------------------------------------------------------------------- verification

def _bruteforce_longest(out, rows_argmax, rows, L):
    """Deepest slot whose every edge matches the target argmax of its parent's row."""
    n = int(out["n_nodes"][0])
    best = (0, [])
    for j in range(1, n):
        chain, b = [], j
        while b > 0:
            chain.append(b)
            b = int(out["par"][0, b])
        chain.reverse()
        ok, prev = True, 0
        for s in chain:
            key = int(out["depth"][0, prev]) if rows == "position" else prev
            if rows == "position" and key >= L:
                ok = False
                break
            if rows_argmax[key] != out["tok"][0, s]:
                ok = False
                break
            prev = s
        if ok and len(chain) > best[0]:
            best = (len(chain), chain)
    return best


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("rows", ["position", "node"])
def test_verify_matches_bruteforce_longest_valid_path(seed, rows):
    inp = tiny_inputs(seed, L=4, V=6, K=3, W=3, B=8, rows=rows)
    out = oracle.build(inp)
    rng = np.random.default_rng(seed)
    L = inp["cfg"].L
    nrow = L if rows == "position" else inp["cfg"].B + 1
    # target rows whose argmax often hits a drafted token
    t = rng.integers(-2, 3, size=(1, nrow, 6)).astype(np.float32)
    for r in range(nrow):
        if rng.random() < 0.7:
            cands = out["tok"][0, 1:int(out["n_nodes"][0])]
            t[0, r, int(rng.choice(cands))] = 9.0
    v = oracle.verify(out, t, "f32", rows, L)
    am = [int(np.argmax(t[0, r])) for r in range(nrow)]
    length, chain = _bruteforce_longest(out, am, rows, L)
    assert v["accepted_len"][0] == length
    assert v["path"][0, :length].tolist() == chain
    assert np.all(v["path"][0, length:] == -1)
    last = chain[-1] if chain else 0
    key = int(out["depth"][0, last]) if rows == "position" else last
    expect_bonus = -1 if (rows == "position" and key >= L) else am[key]
    assert v["bonus"][0] == expect_bonus


def test_verify_full_acceptance_and_immediate_rejection():
    inp = tiny_inputs(4, L=5, V=9, K=3, W=1, B=5)
    out = oracle.build(inp)
    L = 5
    t = np.zeros((1, L, 9), np.float32)
    for d in range(1, L + 1):
        t[0, d - 1, out["tok"][0, d]] = 1.0
    v = oracle.verify(out, t, "f32", "position", L)
    assert v["accepted_len"][0] == L and v["bonus"][0] == -1
    assert v["path"][0].tolist() == list(range(1, L + 1))
    absent = [x for x in range(9) if x != out["tok"][0, 1]][0]
    t[0, 0] = 0.0
    t[0, 0, absent] = 1.0
    v = oracle.verify(out, t, "f32", "position", L)
    assert v["accepted_len"][0] == 0 and v["bonus"][0] == absent


# --------------------------------------------------------------------------- planted mistakes are caught

def _wrong_child_logits(h_par, cand_logit, Ec, Wq):
    H = Wq.shape[0]
    return cand_logit[None, :] + (h_par @ Wq @ Ec.T) / math.sqrt(H)   # W_q transposed


def _wrong_score(s_par, logq, beta):
    return s_par[:, None] + logq                                       # beta dropped


def _wrong_key(score, flat):
    return (-score, -flat)                                             # ties to the higher index


def _wrong_rms(x, eps=od.RMS_EPS):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)    # sum instead of mean


@pytest.mark.parametrize("name,fake", [("child_logits", _wrong_child_logits),
                                       ("score_children", _wrong_score),
                                       ("depth_key", _wrong_key),
                                       ("rmsnorm", _wrong_rms)])
def test_planted_mistakes_fail_the_worked_example(monkeypatch, name, fake):
    monkeypatch.setattr(od, name, fake)
    with pytest.raises(AssertionError):
        test_closed_form_worked_example("f32")
