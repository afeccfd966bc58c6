"""bench.py's accounting on CPU: the weight bytes a step streams (the roofline
numerator's floor) against the generator's actual weight arrays, the metric
names, and the consistency of the workload table."""
import numpy as np
import pytest

import bench
from synthetic import WORKLOADS, gen


def _gemm_weight_bytes(cfg, W):
    """Bytes of every GEMM weight matrix the generator produced (codes for FP8)."""
    def nbytes(a):
        return a.codes.nbytes if hasattr(a, "codes") else np.asarray(a).nbytes
    total = nbytes(W["w_fc"]) + nbytes(W["lm_head"])
    for lw in W["layers"]:
        total += sum(nbytes(lw[k]) for k in ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down"))
        if "conv" in lw:
            total += sum(nbytes(w) for w, _ in lw["conv"].values())
    return total


@pytest.mark.parametrize("name", ["T1", "T1D2", "T1F8", "T1D2F8", "T1S5"])
def test_weight_bytes_match_the_generated_weights(name):
    cfg = WORKLOADS[name].cfg
    W = gen.make_weights(cfg, WORKLOADS[name].seed)
    assert bench.weight_bytes(cfg) == _gemm_weight_bytes(cfg, W)


def test_weight_bytes_of_the_bench_workloads():
    c1, c1f8 = WORKLOADS["C1"].cfg, WORKLOADS["C1F8"].cfg
    assert bench.weight_bytes(c1) == pytest.approx(3.3418e9, rel=1e-3)
    assert bench.weight_bytes(c1f8) == bench.weight_bytes(c1) / 2


def test_metric_names():
    assert bench.metric(WORKLOADS["C1"].cfg) == bench.METRIC
    assert "(5-tok)" in bench.metric(WORKLOADS["C1S5"].cfg)


def test_workload_table_is_consistent():
    for name, wl in WORKLOADS.items():
        c = wl.cfg
        assert 2 <= c.block <= 16, name
        assert len(wl.p_accept) >= c.block - 1, name
        assert c.n_q_heads % c.n_kv_heads == 0 and c.n_q_heads // c.n_kv_heads <= 8, name
        if c.weight_fp8 or c.split_act:
            assert c.dtype == "bf16", name
        if c.weight_fp8:
            assert c.ffn % 16 == 0 and c.feat_in % 16 == 0, name   # one-byte code rows: 16-byte multiples


def _run_bench(*args, env_extra=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) on the tiny
    workload: one JSON line with the contract's keys, no GPU needed."""
    (line,) = _run_bench("--impl", "reference", "--workload", "C0", "--steps", "1", "--warmup", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["warmup"] >= 3 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench("--impl", "reference", "--workload", "C0", "--steps", "1", "--warmup", "1",
                      env_extra={"RANK": "1"}) == []


def test_clock_summary_reads_only_the_timed_region():
    """The nvidia-smi rows inside [t0, t1] plus the first one after: median SM
    clock, max clock, and every throttle reason seen active there."""
    cs = bench.ClockSampler(0)
    na, ac = "Not Active", "Active"

    def row(sm, hw=na, thermal=na, sw_thermal=na, cap=na):
        return ["0", str(sm), "2070", "900.5", "0x0", hw, thermal, sw_thermal, cap]

    cs.rows = [(0.5, row(1000, hw=ac)),                     # before the region: ignored
               (1.1, row(2070)), (1.2, row(1950, cap=ac)), (1.3, row(2070)),
               (2.05, row(1800, sw_thermal=ac)),            # first sample after the end: kept
               (2.5, row(900, thermal=ac))]                 # later: ignored
    cs.t0, cs.t1 = 1.0, 2.0
    s = cs.summary()
    assert s["samples"] == 4
    assert s["sm_mhz"] == 2010.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert bench.ClockSampler(0).summary()["reasons"] == ["unsampled"]


def test_prefill_injection_flops():
    """C1's 2048-token prefill: feature projection 20 480 -> 4 096 plus five
    layers of K and V (8 heads x 128 each) from 4 096: 2 * 2048 * 4096 *
    (20 480 + 5 * 2 * 1024) = 515.4 GFLOP."""
    c1 = WORKLOADS["C1"].cfg
    assert bench.prefill_injection_flops(c1, 2048) == 2.0 * 2048 * 4096 * 30720
    assert bench.prefill_injection_flops(c1, 0) == 0.0
