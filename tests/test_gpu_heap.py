"""The node-by-node heap -> correction baseline (dartree_heap_build) on the GPU.

Blog section 2 (latency breakdown) and section 4.3, Table 2 compare the deferred
search with drafting that pops one node at a time and runs the correction head on
it. The GPU baseline is checked against the oracle's node-by-node search
(oracle.full_tree_heap: a binary heap over the unpruned K-ary tree, the head
evaluated per popped node with scalar loops) pop by pop, and, with W >= B, against
the deferred tree built by dartree_build_tree (the same node set: pin P6).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from dartree_inputs import make_config, make_inputs, make_tie_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    import diffusion_drafter_draft_gb300 as m
    m.lib()
    return m


from _gpu import SCORE_ATOL, upload  # noqa: E402


def _paths(out, i):
    """Token path and score of every pop of request i, in pop order."""
    tok, par, sc = out["tok"][i], out["parent"][i], out["score"][i]
    res = []
    for t in range(len(tok)):
        if tok[t] < 0:
            break
        p, b = [int(tok[t])], int(par[t])
        while b >= 0:
            p.append(int(tok[b]))
            b = int(par[b])
        res.append((tuple(reversed(p)), float(sc[t])))
    return res


@pytest.mark.parametrize("recipe", ["random", "ties"])
@pytest.mark.parametrize("C,L,V,H,K,B,beta", [(2, 4, 3001, 256, 16, 12, -0.1), (1, 5, 2000, 384, 8, 20, -0.05),
                                              (3, 3, 1500, 128, 24, 9, 0.0)])
def test_heap_pops_match_the_oracle(dd, recipe, C, L, V, H, K, B, beta):
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=C, L=L, V=V, H=H, K=K, W=1, B=B, beta=beta, seed=31 * C + K)
    inp = make_tie_inputs(cfg) if recipe == "ties" else make_inputs(cfg)
    x = upload(inp)
    out = dd.heap_build(x["E"], x["Wq"], x["base"], x["hidden"], x["anchor"], K, B, beta)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items() if k != "_keep"}
    for i in range(C):
        want = oracle.full_tree_heap(inp, i, B)
        got = _paths(g, i)
        assert [p for p, _ in got] == [p for p, _ in want], f"request {i}"
        np.testing.assert_allclose([s for _, s in got], [s for _, s in want], rtol=0, atol=SCORE_ATOL)
        d = g["depth"][i]
        assert np.all(d == np.array([len(p) for p, _ in got]))


def test_heap_equals_deferred_tree_when_width_covers_the_budget(dd):
    """Pin P6 on the GPU at the Qwen3-4B shape: with W >= B the deferred tree keeps
    exactly the nodes node-by-node best-first popping reaches."""
    cfg = make_config("cfg1_qwen3_4b_c1").replace(W=64, B=64)
    inp = make_inputs(cfg)
    x = upload(inp)
    heap = dd.heap_build(x["E"], x["Wq"], x["base"], x["hidden"], x["anchor"], cfg.K, cfg.B, cfg.beta)
    tree = dd.build_tree(x["E"], x["Wq"], x["base"], x["hidden"], x["anchor"], cfg.K, cfg.W, cfg.B, cfg.beta)
    torch.cuda.synchronize()
    h = {k: v.cpu().numpy() for k, v in heap.items() if k != "_keep"}
    t = {k: v.cpu().numpy() for k, v in tree.items()}
    got = _paths(h, 0)
    deferred = []
    for j in range(1, int(t["n_nodes"][0])):
        p, b = [], j
        while b > 0:
            p.append(int(t["tok"][0, b]))
            b = int(t["par"][0, b])
        deferred.append((tuple(reversed(p)), float(t["score"][0, j])))
    assert sorted(p for p, _ in got) == sorted(p for p, _ in deferred)
    ds = dict(deferred)
    for p, s in got:
        assert abs(ds[p] - s) <= SCORE_ATOL
