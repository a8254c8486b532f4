"""The key-tile rules shared by the plan and the kernels (csrc/ca_internal.h:
key_tile_ranges, visits_upto, key_tile_rows, key_tile_query_tiles,
key_pair_query_tiles) checked tile by tile against brute-force enumeration of
the visibility rule of include/ca.h on random tasks, with and without masks
(tests/tile_rules_check.cpp, compiled for the host)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path_factory.mktemp("tile_rules") / "tile_rules_check")
    r = subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(cuda, "include"),
                        os.path.join(HERE, "tile_rules_check.cpp"), "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_key_tile_rules_match_brute_force(checker, seed):
    r = subprocess.run([checker, "4000", str(seed)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
