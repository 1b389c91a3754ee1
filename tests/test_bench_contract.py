"""The benchmark's reference arm (the CPU oracle on the host cores) keeps the
JSON-line contract, on the CPU (no GPU): one line, the metric and unit of the
measured arm, the sample it timed, and an end-to-end figure without copies;
under torchrun only rank 0 works and prints."""
import json

import bench


def test_reference_arm_prints_one_contract_line(capsys):
    assert bench.main(["--impl", "reference", "--workload", "1", "--steps", "3",
                       "--warmup", "3"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "us/call"
    assert line["higher_is_better"] is False and line["n_gpus"] == 1
    assert (line["steps"], line["warmup"]) == (3, 3)
    assert line["value"] > 0 and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith("cfg1")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["unit"] == "us/call" and "rows" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "us/call",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_works_on_rank_zero_only(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--workload", "1", "--steps", "3"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_fewer_than_three_warmup_steps_are_raised_to_three(capsys):
    assert bench.main(["--impl", "reference", "--workload", "1", "--steps", "1",
                       "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["warmup"] == 3
