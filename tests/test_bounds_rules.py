"""The range rules of the bounds-checked build, on the host: the pure
functions the checked kernels apply to every access, compiled with nvcc into
a small host program (tests/native/bounds_rules.cu) and compared with
answers worked out by hand. Also: the checked library loads without a GPU
and says it is the checked one. No GPU."""
import os
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# smem_access_ok(offset, bytes, region size): inside, aligned to the size
SMEM = {(0, 16, 128): 1, (112, 16, 128): 1, (116, 16, 128): 0, (128, 16, 128): 0,
        (-16, 16, 128): 0, (124, 4, 128): 1, (126, 4, 128): 0, (128, 4, 128): 0,
        (0, 16, 8): 0}
# grid_access_ok(index, count) on a 6 x 8 array (48 floats)
GRID = {(0, 1): 1, (47, 1): 1, (48, 1): 0, (44, 4): 1, (45, 4): 0, (-1, 1): 0,
        (9, 4): 1, (10, 4): 1}
# interior_access_ok(index, count) for n = 6, ld = 8: rows 1..4, columns 1..4
INTERIOR = {(9, 4): 1,    # row 1, columns 1..4
            (10, 4): 0,   # columns 2..5: 5 is the ring
            (10, 3): 1,   # columns 2..4
            (12, 1): 1,   # column 4
            (13, 1): 0,   # column 5: ring
            (8, 1): 0,    # column 0: ring
            (1, 1): 0,    # row 0: ring
            (41, 1): 0,   # row 5: ring
            (33, 4): 1,   # row 4, columns 1..4
            (14, 1): 0,   # column 6: row padding
            (36, 1): 1,   # row 4, column 4
            (33, 1): 1}
TMA = {0: 1, 4: 1, -4: 1, 2: 0, -3: 0, 1: 0, 120: 1}


@pytest.fixture(scope="module")
def rule_table():
    exe = os.path.join(tempfile.mkdtemp(prefix="tbj_rules_"), "bounds_rules")
    src = os.path.join(ROOT, "tests", "native", "bounds_rules.cu")
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    # the header also holds sm_100-class device code, hence the target
    subprocess.check_call([nvcc, "-std=c++17", "-gencode",
                           "arch=compute_103a,code=sm_103a", "-o", exe, src])
    out = subprocess.check_output([exe], text=True)
    table = {}
    for line in out.splitlines():
        name, *args = line.split()
        table[(name, tuple(int(a) for a in args[:-1]))] = int(args[-1])
    return table


def test_shared_memory_rule(rule_table):
    for k, v in SMEM.items():
        assert rule_table[("smem", k)] == v, k


def test_grid_rule(rule_table):
    for k, v in GRID.items():
        assert rule_table[("grid", k)] == v, k


def test_interior_store_rule(rule_table):
    for k, v in INTERIOR.items():
        assert rule_table[("interior", k)] == v, k


def test_tma_x_rule(rule_table):
    for k, v in TMA.items():
        assert rule_table[("tma", (k,))] == v, k


def test_checked_library_identifies_itself():
    from temporal_blocked_jacobi_gb300 import _build, jacobi
    _build.build_all()
    assert jacobi.load(checked=True).jacobi_bounds_checked() == 1
    assert jacobi.load().jacobi_bounds_checked() == 0
