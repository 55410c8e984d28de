"""The reference arm's oracle steps on CPU (tiny model, host-drawn inputs): whole steps,
and the bounded layer samples it falls back to when whole steps would not fit its time
budget -- the sample's estimate scales the layers' time to every layer."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_oracle_steps_whole_and_sampled():
    import bench
    o = bench.OracleSteps("tiny_b1_64", 0)
    L = o.cfg["n_layers"]
    whole = o.step()
    assert whole > 0
    assert o.step(L) > 0  # every layer: a whole step
    sampled = o.step(1)
    assert sampled > 0
    assert "whole" in o.describe(3) and f"first 1 of {L} layers" in o.describe(3, 1)


def test_reference_line_reports_the_sample(capsys, monkeypatch):
    import json

    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload", "tiny_b1_64",
                                      "--steps", "2", "--warmup", "1"])
    assert bench.main() in (0, None)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and "whole" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
