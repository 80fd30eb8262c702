"""The two-group stream-K split (he::TileSplit in the pipeline header), checked
on the host: compiled with nvcc into a small program that walks every small
shape and every first group the host may choose, plus large random shapes.
The stream kernel takes its tile range from TileSplit::begin and merge finds a
unit's partials with TileSplit::owner, so the two must agree exactly.  CPU
only (host code; no GPU needed)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "lsh_pre_attention_decode_b300", "csrc")


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not found")
def test_tile_split_ranges_and_owners(tmp_path):
    exe = str(tmp_path / "tile_split_check")
    subprocess.run(["nvcc", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-o", exe,
                    os.path.join(HERE, "tile_split_check.cu")], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok "), r.stdout + r.stderr
