"""Host-side arithmetic of bench.py, no GPU: the method's work of each kernel family
over one round (the roofline numerator), the implementation's intermediates
reported beside it, and the roofline of the dominant family (per-launch work =
round work / launches per round, achieved = work / mean launch time)."""
import bench
from dartree_inputs import make_config


def _sum_parents(cfg):
    P, tot = 1, 1
    for _ in range(cfg.L - 1):
        P = min(cfg.W, P * cfg.K)
        tot += P
    return tot


def test_parents_per_depth():
    cfg = make_config("cfg1_qwen3_4b_c1")
    assert bench.parents(cfg) == [1] + [12] * 15
    assert sum(bench.parents(cfg)) == _sum_parents(cfg) == 181


def test_kernel_work_candidate_side_round():
    cfg = make_config("cfg1_qwen3_4b_c1")
    C, L, V, H, K = cfg.C, cfg.L, cfg.V, cfg.H, cfg.K
    # S1 reads the logit rows once; the copied candidate rows are an intermediate
    assert bench.kernel_work(cfg, "topk_rows_kernel", 1.0, True) == ("hbm", C * L * V * 2, 0, 0)
    assert bench.kernel_work(cfg, "topk_rows_kernel", 1.0, True, True) == \
        ("hbm", C * L * V * 2, 2 * C * L * K * H * 2, 0)
    # the G GEMM is charged S3's projection flops; the reassociation's surplus is extra
    bound, work, inter, extra = bench.kernel_work(cfg, "gemm_bf16_tc_kernel", 1.0, True)
    proj = 2 * C * 181 * H * H
    assert bound == "tensor" and work == proj
    assert extra == 2 * C * L * K * H * H - proj
    assert abs(work / 1e9 - 2.37) < 0.01 and abs((work + extra) / 1e9 - 13.42) < 0.01
    assert inter == C * L * K * H * 2 + 2 * C * L * K * H * 2
    # the cluster expansion: candidate rows and block hidden rows (5.32 MB); G is intermediate
    bound, work, inter, extra = bench.kernel_work(cfg, "expand_g_kernel", 1.0, True)
    assert bound == "hbm" and work == C * L * K * H * 2 + C * L * H * 2
    assert abs(work / 1e6 - 5.32) < 0.01
    assert inter >= 2 * C * L * K * H * 2 and extra == 0
    assert bench.kernel_work(cfg, "no_such_kernel", 1.0, True) == ("hbm", 0, 0, 0)


def test_dominant_kernel_roofline_counts_method_bytes():
    cfg = make_config("cfg1_qwen3_4b_c1")
    n = 10
    kt = {"expand_g_kernel": (n, 0.67), "topk_rows_kernel": (n, 0.25), "gemm_bf16_tc_kernel": (n, 0.24)}
    roof, per_kernel, lpr = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 1.0},
                                                  6769.1, 1879.0)
    work = cfg.L * cfg.K * cfg.H * 2 + cfg.L * cfg.H * 2
    assert roof["kernel"] == "expand_g_kernel" and roof["bound"] == "hbm"
    assert roof["bytes_per_launch"] == work
    assert roof["intermediate_bytes_per_launch"] >= 2 * cfg.L * cfg.K * cfg.H * 2
    assert abs(roof["achieved"] - work / 0.067e-3 / 1e9) < 0.01
    assert abs(roof["frac"] - roof["achieved"] / 6769.1) < 1e-4
    assert 0.011 < roof["frac"] < 0.013          # ~0.012 of HBM: latency-bound, not bandwidth-bound
    assert lpr == 3 and list(per_kernel)[0] == "expand_g_kernel"


def test_tensor_bound_gemm_roofline():
    cfg = make_config("cfg1_qwen3_4b_c1")
    n = 4
    kt = {"gemm_bf16_tc_kernel": (n, 0.1), "topk_rows_kernel": (n, 0.08), "expand_g_kernel": (n, 0.05)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 1.0}, 6769.1, 1879.0)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    proj = 2 * 181 * cfg.H * cfg.H
    assert roof["flops_per_launch"] == proj
    assert roof["extra_flops_per_launch"] == 2 * cfg.L * cfg.K * cfg.H * cfg.H - proj
    assert abs(roof["achieved"] - proj / 0.025e-3 / 1e12) < 0.01


def test_concurrent_halves_contraction():
    """From SPLIT_MIN_C requests the expansion runs as two halves on two streams: a
    launch covers half of the batch (32 requests x 512 candidate rows x 8 KB =
    134.2 MB of method bytes), and the whole-batch ncu traffic is halved."""
    cfg = make_config("cfg4_c64_stress")
    assert cfg.C >= bench.SPLIT_MIN_C
    n = 10
    launches = 2 * cfg.L * n
    kt = {"contract_tc_kernel": (launches, 15.8), "gemm_bf16_tc_kernel": (launches, 8.6)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 0.1},
                                       6769.1, 1879.0)
    assert roof["concurrent_halves"] == 2
    assert roof["bytes_per_launch"] == 32 * 512 * 4096 * 2
    assert roof["intermediate_bytes_per_launch"] > 0
    assert roof["traffic"] == bench.NCU_TRAFFIC[("cfg4_c64_stress", "contract_tc_kernel")] // 2
    # 49.2 us per launch would be 0.40 of the measured copy bandwidth
    kt = {"contract_tc_kernel": (launches, launches * 0.04922)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 0.1},
                                       6769.1, 1879.0)
    assert abs(roof["frac"] - 0.403) < 0.002


def test_algorithmic_round_bytes_add_up():
    for name in ("cfg1_qwen3_4b_c1", "cfg4_c64_stress"):
        cfg = make_config(name)
        eb = 2 if cfg.dtype == "bf16" else 4
        a = bench.algorithmic(cfg, 1.0)
        assert a["total"] == a["topk"] + a["expand"] + a["verify"]
        assert a["topk"] == cfg.C * cfg.L * cfg.V * eb
        # W_q once per round; the per-depth variant re-reads it at the other L - 1 depths
        assert a["total_wq_per_depth"] - a["total"] == (cfg.L - 1) * cfg.H * cfg.H * eb
    cfg4 = make_config("cfg4_c64_stress")
    a = bench.algorithmic(cfg4, 0.1)
    assert abs(a["total_wq_per_depth"] / 1e9 - 5.18) < 0.02   # 5.15 GB build + walked rows


def test_both_arms_share_the_config_object():
    cfg = make_config("cfg1_qwen3_4b_c1")
    c = bench.workload_config(cfg, True, 1)
    assert c["workload"] == cfg.name and c["parallelism"] == "single" and c["cuda_graph"] is True
    assert set(c) >= {"C", "L", "V", "H", "K", "W", "B", "beta", "l2"}
    assert bench.workload_config(cfg, True, 4)["parallelism"] == "replicas"


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_every_measurement_the_main_path_calls_exists():
    import ast
    import inspect
    tree = ast.parse(inspect.getsource(bench.main))
    called = {n.func.id for n in ast.walk(tree) if isinstance(n, ast.Call) and isinstance(n.func, ast.Name)}
    missing = [n for n in called if n.startswith(("measure", "kernel_", "roofline", "cpu_", "workload_", "job_"))
               and not hasattr(bench, n)]
    assert not missing, missing
