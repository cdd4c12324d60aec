"""Host-side logic of bench.py (no GPU): the algorithmic bytes and FLOPs the roofline divides
by, the per-format byte sizes, the recorded-traffic lookup and the workload labels."""
import importlib.util
import os

import numpy as np
import pytest

from latent_moe_layer_route_gb300 import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


@pytest.mark.parametrize("fmt,wb,qb", [("fp8", 1.0, 1.0), ("nvfp4", 0.5625, 1.0),
                                       ("mxfp8", 1.03125, 1.03125),
                                       ("nvfp4_w4a4", 0.5625, 0.5625)])
def test_algorithmic_bytes_closed_form(fmt, wb, qb):
    cfg = configs.DECODE_M16.with_(routed_fmt=fmt)
    H, L, I, Is, k, M = cfg.H, cfg.L, cfg.I, cfg.Is, cfg.topk, cfg.M
    cnt = np.zeros(cfg.E, dtype=np.int64)
    cnt[:40] = 1  # 40 experts touched
    ab = bench.algorithmic_bytes(cfg, cnt, M)
    assert ab["touched_experts"] == 40
    routed_w = 40 * 3 * I * L * wb            # W13 (2I x L) and W2 (L x I) of 40 experts
    dense_w = (2 * Is * H + H * Is + H * L) * 2  # bf16 shared expert and up-projection
    gemm = ab["gemm_l1"] + ab["gemm_l2"] + ab["norm"] + ab["gemm_out"]
    # the weights dominate; what remains are token operands and stage outputs
    acts = (M * H * 2 + M * k * L * qb + 2 * M * k * I * qb + M * Is * 2 + M * L * 4
            + M * L * 4 + M * L * 2 + M * L * 2 + M * Is * 2 + M * H * 2)
    assert gemm == pytest.approx(routed_w + dense_w + acts, rel=1e-12)
    assert ab["total"] == pytest.approx(gemm + ab["route"] + ab["perm"], rel=1e-12)


def test_flops_closed_form():
    cfg = configs.PREFILL_M4096
    routed, dense = bench.flops(cfg, cfg.M)
    assert routed == 2.0 * cfg.M * cfg.topk * 3 * cfg.I * cfg.L
    assert dense == 2.0 * cfg.M * (3 * cfg.Is * cfg.H + cfg.H * cfg.L)


def test_dtype_labels_name_each_format():
    labels = {f: bench.dtype_of(configs.DECODE_M16.with_(routed_fmt=f))
              for f in ("fp8", "nvfp4", "mxfp8", "nvfp4_w4a4")}
    assert len(set(labels.values())) == 4
    assert "e2m1" in labels["nvfp4_w4a4"] and "power-of-two" in labels["mxfp8"]


def test_recorded_traffic_only_for_the_recorded_sources():
    dg = bench.kernel_digest()
    assert len(dg) == 16
    for (w, k), (v, d) in bench.NCU_TRAFFIC.items():
        assert bench.recorded_traffic(w, k) == (v if d == dg else None)
    assert bench.recorded_traffic("no_such_workload", "gemm_fused") is None
    # every benchmark workload has an entry (the hidden-state one under its own label)
    names = {w for w, _ in bench.NCU_TRAFFIC}
    assert {c.name for c in configs.ALL} <= names
    assert bench.HEADLINE + "+hidden" in names


def test_job_throughput_counts_every_replica():
    assert bench.job_throughput(1, 16, 10, 1.0) == pytest.approx(160000.0)
    assert bench.job_throughput(4, 16, 10, 1.0) == pytest.approx(640000.0)


def test_launch_names_follow_the_launch_structure():
    d16, mx = configs.DECODE_M16, configs.PREFILL_M4096.with_(routed_fmt="mxfp8")
    assert bench.launch_names(d16, 2, False, False) == ["route_perm", "gemm_fused"]
    assert bench.launch_names(d16, 2, False, True) == ["proj", "route_perm", "gemm_fused"]
    assert bench.launch_names(d16, 5, True, False) == \
        ["route_perm", "gemm_l1", "gemm_l2", "norm", "gemm_out"]
    assert bench.launch_names(configs.DECODE_M128, 4, False, False) == \
        ["route", "perm_scatter", "perm_gather", "gemm_fused"]
    assert bench.launch_names(configs.PREFILL_M4096, 5, False, False) == \
        ["route", "perm_hist", "perm_scatter", "perm_gather", "gemm_fused"]
    assert bench.launch_names(mx, 6, False, False) == \
        ["route", "perm_hist", "perm_scatter", "perm_gather", "gemm_routed", "gemm_dense"]
    assert bench.launch_names(configs.PREFILL_M4096, 8, True, False)[-4:] == \
        ["gemm_l1", "gemm_l2", "norm", "gemm_out"]
