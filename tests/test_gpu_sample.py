"""Parity of verification at a temperature T > 0 (dartree_verify_sample) with the
oracle's Gumbel-max sample-and-match walk, through the C ABI.

Accepted lengths, paths and bonus tokens must be bit-exact: both sides take every
draw in float32 on the same Philox4x32-10 noise, so they can differ only where two
perturbed values lie within rounding of each other (a few units in the last place);
a failure message carries the smallest margin the oracle met.

Trees come from the oracle's build (or, at the 64-request size, from a seeded
random tree with DARTree's slot layout); target rows are seeded noise with large
boosts on tokens the tree carries, so that walks go deep and stop at varied depths.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle import sampling as osm  # noqa: E402
from dartree_inputs import breadth_first_slot_depth, make_config, make_inputs, round_to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_drafter_draft_gb300 as dd
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    dd.lib()


from _gpu import host, t  # noqa: E402


BOOST_P = (0.7, 0.2, 0.1)


def _planted_target(tree, rows_mode, L, V, dtype, seed, T=1.0):
    """Noise rows (sigma 2.5) with a boost on one child token of each row's slot(s):
    per-position row d boosts a depth-(d+1) token of a random root path, per-node
    row j boosts the token of one of slot j's children. Boosts of 22, 15 and 11
    (times T above 1, chosen with probabilities BOOST_P) make a drawn token that of
    the boosted child almost surely, about half the time, and rarely."""
    rng = np.random.default_rng(seed)
    boosts = tuple(np.float32(b * max(1.0, T)) for b in (22.0, 15.0, 11.0))
    n = len(tree["n_nodes"])
    nrow = L if rows_mode == "position" else tree["tok"].shape[1]
    out = np.empty((n, nrow, V), np.uint16 if dtype == "bf16" else np.float32)
    for i in range(n):   # one request at a time: the 64-request rows are 1.3 GB in bf16
        x = rng.standard_normal((nrow, V), dtype=np.float32) * np.float32(2.5)
        nn = int(tree["n_nodes"][i])
        kids = {j: [c for c in range(1, nn) if tree["par"][i, c] == j] for j in range(nn)}
        if rows_mode == "position":
            cur = 0
            for d in range(L):
                if not kids[cur]:
                    break
                cur = int(rng.choice(kids[cur]))
                x[d, int(tree["tok"][i, cur])] += boosts[rng.choice(3, p=BOOST_P)]
        else:
            for j in range(nn):
                if kids[j]:
                    x[j, int(tree["tok"][i, int(rng.choice(kids[j]))])] += boosts[rng.choice(3, p=BOOST_P)]
        out[i] = round_to_bf16_bits(x) if dtype == "bf16" else x
    return out


def _dev_tree(tree):
    return {k: torch.from_numpy(np.ascontiguousarray(tree[k]).astype(np.int32)).cuda()
            for k in ("tok", "par", "depth", "n_nodes")}


def _compare(tree, target, dtype, rows_mode, L, T, seed):
    import diffusion_drafter_draft_gb300 as dd
    mode = dd.ROWS_PER_POSITION if rows_mode == "position" else dd.ROWS_PER_NODE
    g = host(dd.verify_sample(_dev_tree(tree), t(target, dtype), mode, L, T, seed))
    o = osm.verify_sample(tree, target, dtype, rows_mode, L, T, seed)
    for k in ("accepted_len", "path", "bonus"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=f"{k} (smallest draw margin {o['min_margin']:.3g})")
    return o


def _oracle_tree(name, **kw):
    cfg = make_config(name).replace(**kw)
    inp = make_inputs(cfg)
    return cfg, oracle.build(inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows_mode", ["position", "node"])
@pytest.mark.parametrize("T", [1.0, 0.45, 2.0])
@pytest.mark.parametrize("shape", ["ragged", "vocab"])
def test_sampled_verify_matches_oracle(dtype, rows_mode, T, shape):
    if shape == "ragged":   # V not a multiple of 8: odd row starts, scalar heads and tails
        cfg, o = _oracle_tree("cfg0_tiny", C=4, V=1001, dtype=dtype, seed=31)
    else:                   # the full vocabulary of the cfg1 shape (a narrow head keeps the oracle quick)
        cfg, o = _oracle_tree("cfg1_qwen3_4b_c1", C=4, H=256, dtype=dtype, seed=32)
    target = _planted_target(o, rows_mode, cfg.L, cfg.V, dtype, seed=int(T * 100) + len(rows_mode), T=T)
    out = _compare(o, target, dtype, rows_mode, cfg.L, T, seed=0x5EED_0000_0000 + cfg.V)
    assert out["accepted_len"].max() >= 2   # the walks go past the root's children


def test_small_temperature_is_the_greedy_walk():
    import diffusion_drafter_draft_gb300 as dd
    cfg, o = _oracle_tree("cfg1_qwen3_4b_c1", C=3, H=256, seed=33)
    target = _planted_target(o, "position", cfg.L, cfg.V, cfg.dtype, seed=4)
    tr, tg = _dev_tree(o), t(target, cfg.dtype)
    s = host(dd.verify_sample(tr, tg, dd.ROWS_PER_POSITION, cfg.L, 1e-7, 9))
    g = host(dd.verify(tr, tg, dd.ROWS_PER_POSITION, cfg.L))
    for k in ("accepted_len", "path", "bonus"):
        np.testing.assert_array_equal(s[k], g[k], err_msg=k)


def test_equal_seeds_repeat_and_other_seeds_differ():
    import diffusion_drafter_draft_gb300 as dd
    cfg, o = _oracle_tree("cfg0_tiny", C=16, V=1024, seed=34)
    target = np.zeros((16, cfg.L, cfg.V), np.float32)   # flat rows: every draw is pure noise
    tr, tg = _dev_tree(o), t(target, "f32")
    a = host(dd.verify_sample(tr, tg, dd.ROWS_PER_POSITION, cfg.L, 1.0, 123))
    b = host(dd.verify_sample(tr, tg, dd.ROWS_PER_POSITION, cfg.L, 1.0, 123))
    c = host(dd.verify_sample(tr, tg, dd.ROWS_PER_POSITION, cfg.L, 1.0, 123 + (1 << 32)))
    np.testing.assert_array_equal(a["bonus"], b["bonus"])
    assert np.mean(a["bonus"] != c["bonus"]) > 0.5
    o1 = osm.verify_sample(o, target, "f32", "position", cfg.L, 1.0, 123 + (1 << 32))
    np.testing.assert_array_equal(c["bonus"], o1["bonus"])


def _random_tree(cfg, rng):
    """A seeded tree with the slot layout of a DARTree tree (W slots per depth after
    the root, parents one depth up, distinct tokens among siblings)."""
    S = cfg.B + 1
    sd = breadth_first_slot_depth(cfg)
    C = cfg.C
    tok = np.zeros((C, S), np.int64)
    par = np.full((C, S), -1, np.int64)
    for i in range(C):
        tok[i, 0] = rng.integers(cfg.V)
        for j in range(1, S):
            up = np.flatnonzero(sd[:j] == sd[j] - 1)
            par[i, j] = rng.choice(up)
            sib = set(tok[i, 1:j][par[i, 1:j] == par[i, j]])
            while True:
                tk = int(rng.integers(cfg.V))
                if tk not in sib:
                    break
            tok[i, j] = tk
    return dict(tok=tok, par=par, depth=np.tile(sd, (C, 1)), n_nodes=np.full(C, S, np.int64))


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_sampled_verify_at_the_64_request_size(T):
    """The 64-request stress shape (V = 151936, per-node target rows, bf16) through one
    launch over all requests; the oracle checks eight requests (both ends of each half
    of the batch and four inside)."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg4_c64_stress")
    rng = np.random.default_rng(40)
    tree = _random_tree(cfg, rng)
    target = _planted_target(tree, "node", cfg.L, cfg.V, cfg.dtype, seed=41, T=T)
    g = host(dd.verify_sample(_dev_tree(tree), t(target, cfg.dtype), dd.ROWS_PER_NODE, cfg.L, T, 77))
    for i in (0, 5, 17, 31, 32, 45, 58, 63):
        sub = {k: v[i:i + 1] for k, v in tree.items()}
        o = osm.verify_sample(sub, target[i:i + 1], cfg.dtype, "node", cfg.L, T, 77, requests=[i])
        for k in ("accepted_len", "path", "bonus"):
            np.testing.assert_array_equal(g[k][i], o[k][0],
                                          err_msg=f"{k} request {i} (smallest margin {o['min_margin']:.3g})")
    assert g["accepted_len"].max() >= 2
