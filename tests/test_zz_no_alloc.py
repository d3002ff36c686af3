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


def test_static_scratch_rejects_sizes_beyond_its_array(dd):
    L_ = dd.lib()
    C = 1 + (256 * 1024) // (8 * 65)  # one request too many for B+1 = 65 row keys
    p = dd.Params(C, 16, 1, 1, 64, 0.0)
    fake = ctypes.c_void_p(256)
    tree = dd.Tree(256, 256, 256, 256, 256, None, None)
    rc = L_.dartree_verify_static(ctypes.byref(p), ctypes.byref(tree), fake, dd.ROWS_PER_NODE, 1000, dd.BF16, fake,
                                  fake, fake, None)
    assert rc == dd.EUNSUPPORTED
