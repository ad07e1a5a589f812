"""Host logic of bench.py (CPU): the L2 rotation, the launch count it claims,
and the traffic record that is reported only for the sources it was taken on."""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from qmoe_inputs import CONFIGS, expert_fc_bytes  # noqa: E402


def _args(l2):
    return argparse.Namespace(l2=l2)


def test_rotation_keeps_inputs_out_of_the_l2():
    # between two uses of one copy, the other copies stream >= 2 x the L2
    for name in ("decode_int2", "decode_many_expert_int4", "mixed_int3_int4", "prefill_int4"):
        cfg = CONFIGS[name]
        n = bench.replicas_for(cfg, _args("rotate"))
        per = cfg.E * (expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2))
        assert n >= 2
        assert (n - 1) * per >= 2 * bench.L2_BYTES
        assert (n - 2) * per < 2 * bench.L2_BYTES or n == 2   # no more copies than needed
        assert bench.replicas_for(cfg, _args("flush")) == 1


def test_launches_per_step():
    # single launch
    assert bench.launches_per_step(CONFIGS["decode_int2"], 2, 0) == 1
    # T <= 64 on the tensor-core path: route+group, gather, fc1, fc2, combine
    assert bench.launches_per_step(CONFIGS["decode_many_expert_int4"], 1, 0) == 5
    # T > 64 with > 1024 routes: route, group, scatter, fc1 (gathering itself), fc2, combine
    assert bench.launches_per_step(CONFIGS["prefill_int4"], 1, 0) == 6
    # decode-class experts beside the GEMM add one kernel per projection
    assert bench.launches_per_step(CONFIGS["decode_many_expert_int4"], 1, 24) == 7


def test_traffic_is_reported_only_for_the_recorded_sources(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.txt"
    sha = bench.sources_sha()
    rec.write_text(f"fused_decode_kernel decode_int2 {sha} 123\n"
                   f"fused_decode_kernel decode_int2 0000000000000000 456\n"
                   f"gemm_kernel_fc1 prefill_int4 {sha} 789\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.measured_traffic("fused_decode_kernel", "decode_int2") == 123
    assert bench.measured_traffic("gemm_kernel_fc1", "prefill_int4") == 789
    assert bench.measured_traffic("gemm_kernel_fc1", "decode_int2") is None
    rec.write_text("fused_decode_kernel decode_int2 0000000000000000 456\n")
    assert bench.measured_traffic("fused_decode_kernel", "decode_int2") is None


def test_algorithmic_bytes_and_flops():
    cfg = CONFIGS["decode_int2"]
    counts = [1] * cfg.E
    by = bench.algorithmic_bytes(cfg, counts)
    assert by["active"] == cfg.E
    per = expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2)
    # weights of the active experts + x in + out + fp32 logits
    assert by["layer"] == cfg.E * per + 2 * cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4
    fl = bench.algorithmic_flops(CONFIGS["prefill_int4"])
    c = CONFIGS["prefill_int4"]
    R = c.T * c.k
    assert fl["fc1"] == 2.0 * R * c.H * 2 * c.I and fl["fc2"] == 2.0 * R * c.I * c.H
