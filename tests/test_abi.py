"""The C ABI library loads, exports every declared entry point, and rejects bad
arguments on the host (no GPU needed: argument checks run before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    import diffusion_drafter_draft_gb300 as dd
    return dd.lib()


def declared():
    with open(os.path.join(ROOT, "include", "dartree.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"DARTREE_API\s+[\w\s\*]+?\b(dartree_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    import diffusion_drafter_draft_gb300 as dd
    assert declared() == sorted(dd.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared():
        assert hasattr(L, name), name


def test_argument_errors_are_reported_on_the_host(L):
    import diffusion_drafter_draft_gb300 as dd
    P = dd.Params
    fake = ctypes.c_void_p(256)  # never dereferenced: checks fail first
    ws_ok = ctypes.c_void_p(1 << 20)
    p = P(1, 4, 8, 2, 8, -0.1)
    assert L.dartree_workspace_bytes(ctypes.byref(p), 100, 64, dd.F32) > 0
    assert L.dartree_workspace_bytes(ctypes.byref(P(1, 4, 8, 2, 8, 0.5)), 100, 64, dd.F32) == 0   # beta > 0
    assert L.dartree_workspace_bytes(ctypes.byref(P(1, 4, 200, 2, 8, -0.1)), 100, 64, dd.F32) == 0  # K > V
    assert L.dartree_workspace_bytes(ctypes.byref(P(1, 4, 8, 2, 9, -0.1)), 100, 64, dd.F32) == 0   # B > L*W
    assert L.dartree_workspace_bytes(ctypes.byref(p), 100, 60, dd.F32) == 0                        # H % 8
    assert L.dartree_topk(fake, 2, 10, 11, dd.F32, fake, fake, ws_ok, 4096, None) == dd.EINVAL
    assert L.dartree_topk(fake, 2, 10, 5, 7, fake, fake, ws_ok, 4096, None) == dd.EDTYPE
    assert L.dartree_topk(fake, 2, 5000, 2000, dd.F32, fake, fake, ws_ok, 4096, None) == dd.EUNSUPPORTED
    assert L.dartree_topk(fake, 2, 10, 5, dd.F32, fake, fake, ctypes.c_void_p(1 << 20 | 8), 4096, None) \
        == dd.EWORKSPACE
    assert L.dartree_topk(fake, 2, 10, 5, dd.F32, fake, fake, ws_ok, 16, None) == dd.EWORKSPACE
    h = dd.Head()
    assert L.dartree_head_init(ctypes.byref(h), fake, fake, 100, 64, dd.F32) == dd.OK
    assert L.dartree_head_init(ctypes.byref(h), None, fake, 100, 64, dd.F32) == dd.EINVAL
    tree = dd.Tree(256, 256, 256, 256, 256, None, None)
    need = L.dartree_workspace_bytes(ctypes.byref(p), 100, 64, dd.F32)
    assert L.dartree_build_tree(ctypes.byref(h), ctypes.byref(P(1, 4, 8, 2, 8, 0.1)), fake, fake, fake,
                                ctypes.byref(tree), None, None, ws_ok, need, None) == dd.EINVAL
    assert L.dartree_build_tree(ctypes.byref(h), ctypes.byref(p), fake, fake, fake,
                                ctypes.byref(tree), None, None, ws_ok, need - 256, None) == dd.EWORKSPACE
    assert L.dartree_verify(ctypes.byref(p), ctypes.byref(tree), fake, 5, 100, dd.F32, fake, fake, fake, ws_ok,
                            need, None) == dd.EDTYPE
    assert L.dartree_status_string(dd.ETIMEOUT) == b"a bounded device-side wait ran out"
    # bounded-wait self-test: argument checks come before any launch
    assert L.dartree_selftest_wait(ws_ok, 4096, 2, 1000, None) == dd.EINVAL          # which
    assert L.dartree_selftest_wait(ws_ok, 4096, 0, 0, None) == dd.EINVAL             # limit 0
    assert L.dartree_selftest_wait(ws_ok, 4096, 1, 2000000, None) == dd.EINVAL       # limit > 1 s
    assert L.dartree_selftest_wait(ws_ok, 256, 0, 1000, None) == dd.EWORKSPACE       # < 512 bytes
    assert L.dartree_selftest_wait(None, 4096, 0, 1000, None) == dd.EWORKSPACE
    # dartree_round checks like build + verify
    assert L.dartree_round(ctypes.byref(h), ctypes.byref(p), fake, fake, fake, fake, 5, ctypes.byref(tree), fake,
                           fake, fake, ws_ok, need, None) == dd.EDTYPE
    assert L.dartree_round(ctypes.byref(h), ctypes.byref(p), fake, fake, fake, fake, 0, ctypes.byref(tree), fake,
                           fake, fake, ws_ok, need - 256, None) == dd.EWORKSPACE


def test_host_session_arguments_are_checked_on_the_host(L):
    """dartree_host_session_create rejects null pointers, an unknown row mode or
    dtype, and shapes dartree_round would reject, before any CUDA call; stage,
    round and input_bytes reject a null session."""
    import diffusion_drafter_draft_gb300 as dd
    P = dd.Params
    fake = ctypes.c_void_p(256)  # never dereferenced: checks fail first
    h = dd.Head()
    assert L.dartree_head_init(ctypes.byref(h), fake, fake, 100, 64, dd.F32) == dd.OK
    p = P(1, 4, 8, 2, 8, -0.1)
    s = ctypes.c_void_p()
    create = L.dartree_host_session_create
    assert create(None, ctypes.byref(p), dd.ROWS_PER_POSITION, ctypes.byref(s)) == dd.EINVAL
    assert create(ctypes.byref(h), None, dd.ROWS_PER_POSITION, ctypes.byref(s)) == dd.EINVAL
    assert create(ctypes.byref(h), ctypes.byref(p), dd.ROWS_PER_POSITION, None) == dd.EINVAL
    assert create(ctypes.byref(h), ctypes.byref(p), 5, ctypes.byref(s)) == dd.EDTYPE
    bad = dd.Head()
    ctypes.memmove(ctypes.byref(bad), ctypes.byref(h), ctypes.sizeof(h))
    bad.dtype = 7
    assert create(ctypes.byref(bad), ctypes.byref(p), dd.ROWS_PER_POSITION, ctypes.byref(s)) == dd.EDTYPE
    assert create(ctypes.byref(h), ctypes.byref(P(0, 4, 8, 2, 8, -0.1)), dd.ROWS_PER_NODE, ctypes.byref(s)) == dd.EINVAL
    assert create(ctypes.byref(h), ctypes.byref(P(1, 4, 8, 2, 8, 0.5)), dd.ROWS_PER_NODE, ctypes.byref(s)) == dd.EINVAL
    assert create(ctypes.byref(h), ctypes.byref(P(1, 4, 200, 2, 8, -0.1)), dd.ROWS_PER_NODE, ctypes.byref(s)) \
        == dd.EINVAL  # K > V
    assert not s.value
    hi, ho = dd.HostInputs(256, 256, 256, 256), dd.HostOutputs(256, 256, 256)
    assert L.dartree_host_stage(None, ctypes.byref(hi)) == dd.EINVAL
    assert L.dartree_host_round(None, ctypes.byref(ho), None) == dd.EINVAL
    assert L.dartree_host_input_bytes(None, 0) == 0
    L.dartree_host_session_destroy(None)  # a null session is ignored


def test_heap_search_limits_are_checked_on_the_host(L):
    import diffusion_drafter_draft_gb300 as dd
    P = dd.Params
    ok = P(2, 4, 16, 1, 12, -0.1)
    assert L.dartree_heap_workspace_bytes(ctypes.byref(ok), 3001, 256, dd.BF16) > 0
    assert L.dartree_heap_workspace_bytes(ctypes.byref(ok), 3001, 256, dd.F32) == 0                 # bf16 only
    assert L.dartree_heap_workspace_bytes(ctypes.byref(P(2, 4, 65, 1, 12, -0.1)), 3001, 256, dd.BF16) == 0  # K
    assert L.dartree_heap_workspace_bytes(ctypes.byref(P(2, 4, 16, 1, 257, -0.1)), 3001, 256, dd.BF16) == 0  # B
    assert L.dartree_heap_workspace_bytes(ctypes.byref(P(2, 4, 16, 1, 12, 0.5)), 3001, 256, dd.BF16) == 0  # beta
    assert L.dartree_heap_workspace_bytes(ctypes.byref(ok), 3001, 200, dd.BF16) == 0                  # H % 128
    fake = ctypes.c_void_p(256)
    head = dd.Head(256, 256, 3001, 256, dd.F32, None)
    assert L.dartree_heap_build(ctypes.byref(head), ctypes.byref(ok), fake, fake, fake, fake, fake, fake, fake,
                                fake, 1 << 20, None) == dd.EUNSUPPORTED
    head = dd.Head(256, 256, 3001, 256, dd.BF16, None)   # not prepared (no W_q^T)
    assert L.dartree_heap_build(ctypes.byref(head), ctypes.byref(ok), fake, fake, fake, fake, fake, fake, fake,
                                fake, 1 << 20, None) == dd.EINVAL


def test_sampled_verify_arguments_are_checked_on_the_host(L):
    import diffusion_drafter_draft_gb300 as dd
    p = dd.Params(1, 4, 8, 2, 8, -0.1)
    fake = ctypes.c_void_p(256)
    ws_ok = ctypes.c_void_p(1 << 20)
    tree = dd.Tree(256, 256, 256, 256, 256, None, None)
    f = L.dartree_verify_sample
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert f(ctypes.byref(p), ctypes.byref(tree), fake, 0, 100, dd.F32, T, 1, fake, fake, fake, ws_ok, 4096,
                 None) == dd.EINVAL
    assert f(ctypes.byref(p), ctypes.byref(tree), fake, 5, 100, dd.F32, 1.0, 1, fake, fake, fake, ws_ok, 4096,
             None) == dd.EDTYPE
    assert f(ctypes.byref(p), ctypes.byref(tree), fake, 0, 100, dd.F32, 1.0, 1, fake, fake, fake, ws_ok, 64,
             None) == dd.EWORKSPACE
    assert f(ctypes.byref(dd.Params(0, 4, 8, 2, 8, -0.1)), ctypes.byref(tree), fake, 0, 100, dd.F32, 1.0, 1, fake,
             fake, fake, ws_ok, 64, None) == dd.OK   # an empty batch launches nothing


def test_adaptive_budget_matches_the_oracle_policy(L):
    import diffusion_drafter_draft_gb300 as dd
    from oracle.sampling import adaptive_budget
    for C in (1, 2, 3, 4, 5, 8, 64, 1000):
        assert dd.adaptive_budget(C) == adaptive_budget(C)
    with pytest.raises(dd.DartreeError):
        dd.adaptive_budget(0)


def test_lm_head_arguments_are_checked_on_the_host(L):
    import diffusion_drafter_draft_gb300 as dd
    fake = ctypes.c_void_p(256)
    ws_ok = ctypes.c_void_p(1 << 20)
    need = L.dartree_lm_head_workspace_bytes(16, 151936, 2560, 64)
    assert need >= 256 + 16 * 64 * 8    # status word + one K-key list per row and SM
    assert L.dartree_lm_head_workspace_bytes(16, 1000, 100, 8) == 0      # H % 64
    assert L.dartree_lm_head_workspace_bytes(16, 1000, 128, 129) == 0    # K > 128
    assert L.dartree_lm_head_workspace_bytes(16, 10, 128, 11) == 0       # K > V
    f = L.dartree_lm_head_topk
    assert f(fake, fake, 16, 1000, 128, 8, dd.F32, fake, fake, ws_ok, need, None) == dd.EUNSUPPORTED
    assert f(fake, fake, 16, 1000, 128, 8, 9, fake, fake, ws_ok, need, None) == dd.EDTYPE
    assert f(fake, fake, 16, 1000, 128, 2000, dd.BF16, fake, fake, ws_ok, need, None) == dd.EINVAL
    assert f(fake, fake, 16, 1000, 100, 8, dd.BF16, fake, fake, ws_ok, need, None) == dd.EUNSUPPORTED
    assert f(ctypes.c_void_p(258), fake, 16, 1000, 128, 8, dd.BF16, fake, fake, ws_ok, 1 << 24, None) \
        == dd.EINVAL                                                     # hidden not 16-byte aligned
    small = L.dartree_lm_head_workspace_bytes(16, 1000, 128, 8)
    assert f(fake, fake, 16, 1000, 128, 8, dd.BF16, fake, fake, ws_ok, small - 8, None) == dd.EWORKSPACE
    assert f(fake, fake, 0, 1000, 128, 8, dd.BF16, fake, fake, ws_ok, 0, None) == dd.OK


def test_tree_attention_limits_are_checked_on_the_host(L):
    import diffusion_drafter_draft_gb300 as dd
    P = dd.AttnParams
    ws = L.dartree_tree_attention_workspace_bytes
    assert ws(ctypes.byref(P(1, 65, 32, 8, 128, 2048, 1e6))) > 0
    assert ws(ctypes.byref(P(1, 65, 32, 8, 64, 2048, 1e6))) == 0     # D != 128
    assert ws(ctypes.byref(P(1, 129, 4, 2, 128, 2048, 1e6))) == 0    # S > 128
    assert ws(ctypes.byref(P(1, 65, 32, 4, 128, 2048, 1e6))) == 0    # 8 heads x 65 slots > 384 rows
    assert ws(ctypes.byref(P(1, 65, 30, 8, 128, 2048, 1e6))) == 0    # Hq not a multiple of Hkv
    assert ws(ctypes.byref(P(1, 65, 32, 8, 128, 2047, 1e6))) == 0    # N % 8
    assert ws(ctypes.byref(P(1, 65, 32, 8, 128, 2048, 0.0))) == 0    # theta
    fake = ctypes.c_void_p(256)
    tree = dd.Tree(None, None, None, None, 256, 256, 256)
    p = P(1, 65, 32, 8, 128, 2048, 1e6)
    need = ws(ctypes.byref(p))
    f = L.dartree_tree_attention
    args = [fake] * 6
    assert f(ctypes.byref(P(1, 65, 32, 8, 64, 2048, 1e6)), *args, ctypes.byref(tree), fake, ctypes.c_void_p(1 << 20),
             need, None) == dd.EUNSUPPORTED
    assert f(ctypes.byref(p), ctypes.c_void_p(264), *args[1:], ctypes.byref(tree), fake, ctypes.c_void_p(1 << 20),
             need, None) == dd.EINVAL                                  # q not 16-byte aligned
    assert f(ctypes.byref(p), *args, ctypes.byref(tree), fake, ctypes.c_void_p(1 << 20), need - 256, None) \
        == dd.EWORKSPACE
    assert f(ctypes.byref(P(0, 65, 32, 8, 128, 2048, 1e6)), *args, ctypes.byref(tree), fake, None, 0, None) == dd.OK


def test_every_kernel_family_has_a_timing_name(L):
    import diffusion_drafter_draft_gb300 as dd
    n = dd.num_kernel_ids()
    names = [L.dartree_kernel_name(k).decode() for k in range(n)]
    assert names[-1] == "other" and len(set(names)) == n
    for want in ("expand_g_kernel", "lmhead_topk_kernel", "attn_kernel", "rowsample_kernel", "heap_search_kernel"):
        assert want in names
    assert L.dartree_kernel_name(n).decode() == "unknown"
