"""The bench's reference arm runs on the host cores: its JSON line keeps the contract."""

import io
import json
from contextlib import redirect_stdout


def test_reference_arm_prints_one_contract_line():
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["n_gpus"] == 1 and j["steps"] == 2 and j["warmup"] == 1
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT and j["higher_is_better"] is True
    assert j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["h2d_bytes_per_step"] == 0
    assert j["config"]["workload"] == bench.WORKLOAD_NAME


def test_traffic_record_is_reported_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """The roofline's `traffic` comes from the committed ncu record and is dropped (None) as soon as
    any of the kernel's source files differs from the one the record was taken on."""
    import bench
    csrc = tmp_path / "verify_bs_step_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.h").write_text("header b\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"sources": ["a.cu", "b.h"], "source_sha": bench.source_sha("a.cu", "b.h"), "dram_bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"bs_step_kernel": rec}))
    assert bench.recorded_traffic("bs_step_kernel")["dram_bytes_per_launch"] == 123
    assert bench.recorded_traffic("another_kernel") is None
    (csrc / "b.h").write_text("header b, changed\n")
    assert bench.recorded_traffic("bs_step_kernel") is None


def test_committed_traffic_record_names_existing_sources():
    import bench
    import os
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))["bs_step_kernel"]
    for name in rec["sources"]:
        assert os.path.exists(os.path.join(bench.ROOT, "verify_bs_step_gb300", "csrc", name)), name
    assert rec["dram_bytes_per_launch"] > 65_667_072       # at least the logits of one Llama-shaped step
