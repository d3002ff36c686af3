"""dartree_verify_static: verification for callers that cannot allocate device memory.

A serving loop whose caching allocator has taken all free HBM, or a plugin behind a
plain C interface, cannot hand this library a workspace. dartree_verify_static keeps
its scratch in a fixed device array instead. These tests call it through the C ABI
and check, on two calls in a row, that it returns exactly what dartree_verify (the
workspace variant) returns. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dartree_inputs import breadth_first_slot_depth, make_config, make_inputs, make_target_per_node  # noqa: E402

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


def _dev(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _case(dd, rows, dtype):
    cfg = make_config("cfg0_tiny").replace(C=3, dtype=dtype, target="argmax", agree_p=0.9, rows=rows, seed=11)
    inp = make_inputs(cfg)
    x = {k: _dev(inp[k], dtype) for k in ("E", "Wq", "base", "hidden")}
    anchor = torch.from_numpy(inp["anchor"]).cuda()
    tree = dd.build_tree(x["E"], x["Wq"], x["base"], x["hidden"], anchor, cfg.K, cfg.W, cfg.B, cfg.beta)
    if rows == "position":
        target, mode = _dev(inp["target"], dtype), dd.ROWS_PER_POSITION
    else:
        target = _dev(make_target_per_node(cfg, inp, breadth_first_slot_depth(cfg)), dtype)
        mode = dd.ROWS_PER_NODE
    return cfg, tree, target, mode


@pytest.mark.parametrize("rows", ["position", "node"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_static_scratch_verify_matches_workspace_verify(dd, rows, dtype):
    cfg, tree, target, mode = _case(dd, rows, dtype)
    ref = dd.verify(tree, target, mode, cfg.L)
    for _ in range(2):  # the array keeps the previous call's contents
        got = dd.verify_static(tree, target, mode, cfg.L)
        torch.cuda.synchronize()
        for k in ("accepted_len", "path", "bonus"):
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=k)


def _random_trees(rng, C, L, B):
    """Valid trees (slot 0 = root, parents earlier and one depth up, n_nodes in 1..B+1)."""
    S = B + 1
    tok = np.full((C, S), -1, np.int32)
    par = np.full((C, S), -1, np.int32)
    depth = np.full((C, S), -1, np.int32)
    n = rng.integers(1, S + 1, size=C).astype(np.int32)
    for i in range(C):
        tok[i, 0], depth[i, 0] = 7, 0
        for j in range(1, int(n[i])):
            cand = [q for q in range(j) if depth[i, q] < L]
            p = int(cand[rng.integers(0, len(cand))])
            par[i, j], depth[i, j], tok[i, j] = p, depth[i, p] + 1, int(rng.integers(0, 64))
    return {k: torch.from_numpy(v).cuda() for k, v in dict(tok=tok, par=par, depth=depth, n_nodes=n).items()}


@pytest.mark.parametrize("rows", ["position", "node"])
def test_static_scratch_accepts_its_exact_limit(dd, rows):
    """C = 503 requests with B + 1 = 65 slots is the largest batch whose row keys
    fit the array (256 + 8 * 503 * 65 <= 256 KiB): accepted, and equal to the
    workspace variant on two calls in a row."""
    C, L, B, V = 503, 16, 64, 64
    assert 256 + 8 * C * (B + 1) <= 256 * 1024 < 256 + 8 * (C + 1) * (B + 1)
    rng = np.random.default_rng(5)
    tree = _random_trees(rng, C, L, B)
    nrow = L if rows == "position" else B + 1
    # small integer logits: argmax ties are frequent, the lowest id must win
    target = torch.from_numpy(rng.integers(-4, 5, size=(C, nrow, V)).astype(np.float32)).cuda().to(torch.bfloat16)
    mode = dd.ROWS_PER_POSITION if rows == "position" else dd.ROWS_PER_NODE
    ref = dd.verify(tree, target, mode, L)
    for _ in range(2):
        got = dd.verify_static(tree, target, mode, L)
        torch.cuda.synchronize()
        for k in ("accepted_len", "path", "bonus"):
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=k)


def test_static_scratch_rejects_sizes_beyond_its_array(dd):
    """One request more than the limit (C = 504 with B + 1 = 65 slots) is rejected
    on the host, before anything is enqueued (the fake pointers are never used)."""
    L_ = dd.lib()
    C = 1 + (256 * 1024 - 256) // (8 * 65)
    assert C == 504
    fake = ctypes.c_void_p(256)
    tree = dd.Tree(256, 256, 256, 256, 256, None, None)
    for rows, L in ((dd.ROWS_PER_NODE, 16), (dd.ROWS_PER_POSITION, 16), (dd.ROWS_PER_POSITION, 64)):
        p = dd.Params(C, L, 1, 1, 64, 0.0)
        rc = L_.dartree_verify_static(ctypes.byref(p), ctypes.byref(tree), fake, rows, 1000, dd.BF16, fake,
                                      fake, fake, None)
        assert rc == dd.EUNSUPPORTED
