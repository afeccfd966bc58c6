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
