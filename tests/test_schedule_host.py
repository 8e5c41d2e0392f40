"""The logits work split (the schedule header's cost model and item iteration), built
for the CPU: every tile of every group goes to exactly one CTA, in order."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_tile_claimed_once(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    exe = str(tmp_path / "schedule_split")
    subprocess.run([cxx, "-std=c++17", "-O1", "-o", exe, os.path.join(HERE, "host", "schedule_split.cpp")],
                   check=True)
    for seed in (1, 2, 3):
        out = subprocess.run([exe, str(seed), "300"], check=True, capture_output=True, text=True).stdout
        assert out.strip() == "OK 300", out
