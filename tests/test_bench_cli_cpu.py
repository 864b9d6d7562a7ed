"""The benchmark's command-line options and result file, on CPU (no GPU call)."""
import argparse
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_emit_prints_and_writes_the_line(tmp_path, capsys):
    line = {"metric": "m", "value": 1.5, "config": {"seed": 3}}
    bench.emit(line, argparse.Namespace(results_dir=str(tmp_path / "res")), "step")
    printed = capsys.readouterr().out.strip()
    assert json.loads(printed) == line
    files = os.listdir(tmp_path / "res")
    assert len(files) == 1 and files[0].startswith("step_") and files[0].endswith(".json")
    assert json.loads((tmp_path / "res" / files[0]).read_text()) == line


def test_emit_without_results_dir_writes_nothing(tmp_path, capsys, monkeypatch):
    monkeypatch.chdir(tmp_path)
    bench.emit({"v": 1}, argparse.Namespace(results_dir=None), "step")
    assert json.loads(capsys.readouterr().out) == {"v": 1}
    assert os.listdir(tmp_path) == []


def test_bad_split_count_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--splits", "0"],
                       capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 2 and "--splits must be >= 1" in r.stderr
