"""Host-side arithmetic of bench.py, no GPU: the algorithmic work of each kernel
family over one round and the roofline of the dominant one (per-launch work =
round work / launches per round, achieved = work / mean launch time)."""
import bench
from dartree_inputs import make_config


def test_kernel_work_cfg1_fused_top_k():
    cfg = make_config("cfg1_qwen3_4b_c1")
    C, L, V, H, K = cfg.C, cfg.L, cfg.V, cfg.H, cfg.K
    # the cluster top-K alone reads the logit rows once
    assert bench.kernel_work(cfg, "topk_rows_kernel", 1.0, True) == ("hbm", C * L * V * 2)
    # in a round it also copies E[cand] (read + write) and reads the target rows
    bound, b = bench.kernel_work(cfg, "topk_rows_kernel", 1.0, True, True, True)
    assert bound == "hbm" and b == 2 * C * L * V * 2 + 2 * C * L * K * H * 2
    assert abs(b / 1e6 - 20.2) < 0.1  # the figure quoted for cfg1
    # G = E[cand] W_q: one tensor-core GEMM over all C*L*K candidate rows
    assert bench.kernel_work(cfg, "gemm_bf16_tc_kernel", 1.0, True) == ("tensor", 2 * C * L * K * H * H)
    assert bench.kernel_work(cfg, "expand_g_kernel", 1.0, True) == ("hbm", 3 * C * L * K * H * 2 + C * L * H * 2)
    assert bench.kernel_work(cfg, "no_such_kernel", 1.0, True) == ("hbm", 0)


def test_kernel_roofline_picks_the_dominant_kernel():
    cfg = make_config("cfg1_qwen3_4b_c1")
    n = 10
    kt = {"expand_g_kernel": (n, 0.67), "topk_rows_kernel": (n, 0.25), "gemm_bf16_tc_kernel": (n, 0.24),
          "finish_kernel": (n, 0.12)}
    roof, per_kernel, lpr = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 1.0},
                                                  6794.5, 1913.9)
    work = 3 * cfg.L * cfg.K * cfg.H * 2 + cfg.L * cfg.H * 2
    assert roof["kernel"] == "expand_g_kernel" and roof["bound"] == "hbm"
    assert roof["bytes_per_launch"] == work
    assert abs(roof["achieved"] - work / 0.067e-3 / 1e9) < 0.01
    assert abs(roof["frac"] - roof["achieved"] / 6794.5) < 1e-4
    assert roof["traffic"] == bench.NCU_TRAFFIC[("cfg1_qwen3_4b_c1", "expand_g_kernel")]
    assert lpr == 4 and list(per_kernel)[0] == "expand_g_kernel"


def test_kernel_roofline_tensor_bound_and_fused_top_k():
    cfg = make_config("cfg1_qwen3_4b_c1")
    n = 4
    # (the candidate-side path is recognised by its expansion kernel in the list)
    kt = {"gemm_bf16_tc_kernel": (n, 0.1), "topk_rows_kernel": (n, 0.08), "expand_g_kernel": (n, 0.05)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 1.0}, 6794.5, 1913.9)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    flops = 2 * cfg.L * cfg.K * cfg.H * cfg.H
    assert roof["flops_per_launch"] == flops
    assert abs(roof["achieved"] - flops / 0.025e-3 / 1e12) < 0.01
    # with no gather or row-max launch in the list, the top-K carries their bytes
    kt = {"topk_rows_kernel": (n, 0.1), "expand_g_kernel": (n, 0.01)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 1.0}, 6794.5, 1913.9)
    assert roof["kernel"] == "topk_rows_kernel"
    assert roof["bytes_per_launch"] == 2 * cfg.L * cfg.V * 2 + 2 * cfg.L * cfg.K * cfg.H * 2


def test_kernel_roofline_concurrent_halves():
    """From SPLIT_MIN_C requests the expansion runs as two halves on two streams: a
    launch covers half of the batch, and the whole-batch ncu traffic is halved."""
    cfg = make_config("cfg4_c64_stress")
    assert cfg.C >= bench.SPLIT_MIN_C
    n = 10
    launches = 2 * cfg.L * n
    kt = {"contract_tc_kernel": (launches, 15.8), "gemm_bf16_tc_kernel": (launches, 8.6)}
    roof, _, _ = bench.kernel_roofline(cfg, {"kernel_times": kt, "n_prof": n, "accepted_mean": 0.1},
                                       6794.5, 1913.9)
    _, round_bytes = bench.kernel_work(cfg, "contract_tc_kernel", 0.1, False)
    assert roof["concurrent_halves"] == 2
    assert roof["bytes_per_launch"] == int(round_bytes / (2 * cfg.L))
    assert roof["traffic"] == bench.NCU_TRAFFIC[("cfg4_c64_stress", "contract_tc_kernel")] // 2


def test_algorithmic_round_bytes_add_up():
    for name in ("cfg1_qwen3_4b_c1", "cfg4_c64_stress"):
        cfg = make_config(name)
        a = bench.algorithmic(cfg, 1.0)
        assert a["total"] == a["topk"] + a["expand"] + a["verify"]
        assert a["topk"] == cfg.C * cfg.L * cfg.V * (2 if cfg.dtype == "bf16" else 4)
