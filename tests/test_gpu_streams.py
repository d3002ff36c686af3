"""Two callers on two streams at the C=64 stress shape.

Each dartree_round call of a 64-request batch forks the second half of its
expansion onto a library side stream that belongs to the caller's stream; two
callers on two streams therefore run concurrently without sharing a side stream.
Both rounds, enqueued back to back on their own streams several times, must give
exactly the trees and verification results of dartree_build_tree followed by
dartree_verify on the default stream (which the other parity tests check against
the oracle).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dartree_inputs import make_config, make_inputs  # noqa: E402

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def test_two_streams_run_c64_rounds_concurrently(dd):
    cfg = make_config("cfg4_c64_stress").replace(rows="position")
    inp = make_inputs(cfg)
    E, Wq = _dev(inp["E"]), _dev(inp["Wq"])
    a = dict(base=_dev(inp["base"]), hidden=_dev(inp["hidden"]), anchor=torch.from_numpy(inp["anchor"]).cuda(),
             target=_dev(inp["target"]))
    # the second caller's batch: the same requests in reverse order
    b = {k: v.flip(0).contiguous() for k, v in a.items()}
    mode = dd.ROWS_PER_POSITION

    def reference(x):
        t = dd.build_tree(E, Wq, x["base"], x["hidden"], x["anchor"], cfg.K, cfg.W, cfg.B, cfg.beta)
        v = dd.verify(t, x["target"], mode, cfg.L)
        torch.cuda.synchronize()
        return {k: t[k].cpu().numpy() for k in ("tok", "par", "depth", "score", "n_nodes", "mask", "pos")}, \
            {k: w.cpu().numpy() for k, w in v.items()}

    ref_a, vref_a = reference(a)
    ref_b, vref_b = reference(b)
    # the reversed batch gives the reversed results
    for k in ref_a:
        np.testing.assert_array_equal(ref_b[k], ref_a[k][::-1], err_msg=k)

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ra = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, mode)
    rb = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, mode)
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            out_a = ra.run(a["base"], a["hidden"], a["anchor"], a["target"])
        with torch.cuda.stream(s2):
            out_b = rb.run(b["base"], b["hidden"], b["anchor"], b["target"])
    torch.cuda.synchronize()
    assert dd.read_status(ra.ws) == 0 and dd.read_status(rb.ws) == 0
    for r, out, ref, vref in ((ra, out_a, ref_a, vref_a), (rb, out_b, ref_b, vref_b)):
        for k in ref:
            np.testing.assert_array_equal(r.tree[k].cpu().numpy(), ref[k], err_msg=k)
        for k in vref:
            np.testing.assert_array_equal(out[k].cpu().numpy(), vref[k], err_msg=k)
