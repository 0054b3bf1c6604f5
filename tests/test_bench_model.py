"""CPU checks of bench.py's measurement arithmetic: the byte model behind the
roofline fraction, the traffic record lookup, the clock record parsing, and the
sampled-unit comparison with the oracle that guards every printed line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_long_sequence_gb300 import workloads  # noqa: E402
from tests import golden  # noqa: E402


def test_byte_model_on_the_text_workload():
    # the text workload's edge count (tests/golden/edge_counts.txt) in the model the
    # roofline fraction divides: per unit and hop 4 E (A read) + the hop state and V
    # traffic; E = 2,271,946, n = 4096, d = 64, bf16 I/O, K = 5, 24 units
    E = golden.edge_counts()["text_bf16_b2h12_n4096"]["total"]
    m = bench.algorithmic_bytes(workloads.TEXT, E)
    per_unit_hops = 4 * E * 5 + 2 * 4096 * 64 * 2 + 4 * (8 * 4096 * 64 + 4096 * 64 * 2)
    assert per_unit_hops == 56_973_256
    assert m["hops_total"] == 24 * per_unit_hops
    assert abs(m["per_hop_launch"] - 273_471_628.8) < 1e-3
    # the whole forward: Q, K, V, out once, A written once and read K times, the hop
    # state between hops, the graph once
    assert m["total"] == 1_619_751_344


def test_byte_model_scales_with_units_and_edges():
    w = workloads.TEXT
    a, b = bench.algorithmic_bytes(w, 1000), bench.algorithmic_bytes(w, 2000)
    # every hop reads each edge's weight once: 4 bytes per edge per hop per unit
    assert b["per_hop_launch"] - a["per_hop_launch"] == 4 * 1000 * w.units
    assert b["total"] - a["total"] == 1000 * (4 * (1 + w.hops) * w.units + 4)


def test_traffic_record_applies_only_to_the_recorded_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "sparse_long_sequence_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.BAND_FILES:
        (csrc / name).write_text("// " + name + "\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha(bench.BAND_FILES)
    rec = {"text_bf16_b2h12_n4096": {"bytes_per_hop": 123456, "source_sha": sha}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.hop_kernel_traffic("text_bf16_b2h12_n4096", "band") == 123456.0
    assert bench.hop_kernel_traffic("lra_bf16_b32h8_n1024", "band") is None      # not recorded
    (csrc / "band_hop.cu").write_text("// changed\n")                             # a kernel edit
    assert bench.hop_kernel_traffic("text_bf16_b2h12_n4096", "band") is None
    # the hash covers names and contents, in a fixed order
    assert bench.kernel_source_sha(tuple(reversed(bench.BAND_FILES))) == bench.kernel_source_sha(bench.BAND_FILES)


def test_clock_record_parsing(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2062, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbage line",
            "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")

    class Done:                     # stands for the finished nvidia-smi process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    s.proc, s.fh = Done(), open(os.devnull, "w")
    rec = s.stop()
    assert rec == {"sm_mhz": 2062.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(s.path)


def test_clock_record_reports_throttling(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("0, 1500, 2070, 1400, 0x8, Active, Not Active, Active, Not Active\n")

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    s.proc, s.fh = Done(), open(os.devnull, "w")
    assert s.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def _unit_reference(w, Qh, Kh, Vh, unit):
    import oracle
    b, h = divmod(unit, w.H)
    row_ptr, col = oracle.token_graph(**w.graph_args(), causal=w.kind == "causal")
    one = [oracle.widen(x[b:b + 1, h:h + 1], w.dtype) for x in (Qh, Kh, Vh)]
    return oracle.forward(*one, row_ptr, col, w.hops, w.alpha)[0, 0]


def test_sampled_unit_check_fires_on_a_wrong_output():
    import pytest
    from sparse_long_sequence_gb300 import synthetic
    for w, bump in ((workloads.BY_NAME["tiny_fp32_n512"], 2e-5), (workloads.BY_NAME["lra_bf16_b32h8_n1024"], 6e-3)):
        Qh, Kh, Vh = synthetic.qkv(w.B, w.H, w.n, w.d, w.dtype, seed=w.seed)
        unit = w.units - 1
        ref = _unit_reference(w, Qh, Kh, Vh, unit)
        ok = bench.check_sampled_unit(w, ref, Qh, Kh, Vh, unit)
        assert ok["error"] == 0.0 and ok["unit"] == unit
        bad = ref.copy()
        bad[7, 3] += bump * (1.0 if w.dtype == "fp32" else abs(ref[7]).max())
        with pytest.raises(bench.BenchCheckFailed):
            bench.check_sampled_unit(w, bad, Qh, Kh, Vh, unit)
