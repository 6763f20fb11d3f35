"""The C-ABI library builds for sm_103a, loads without a GPU, and exports
every function include/jacobi.h declares (no compute calls here)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "jacobi.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jacobi_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("jacobi_create", "jacobi_rhs", "jacobi_solve_step",
                     "jacobi_residual", "jacobi_destroy", "jacobi_set_strategy",
                     "jacobi_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol():
    from temporal_blocked_jacobi_gb300 import _build
    path = _build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_defaults_without_gpu():
    from temporal_blocked_jacobi_gb300 import jacobi
    lib = jacobi.load()
    assert lib.jacobi_status_string(-3) == b"JACOBI_ERR_NOT_CONVERGED"
    cfg = jacobi.make_config()
    assert (cfg.strategy, cfg.depth, cfg.check_every, cfg.tol, cfg.max_sweeps) == \
        (jacobi.SYNC, 1, 8, 1e-5, 1 << 22)
    assert ctypes.sizeof(jacobi.Config) == 64


def test_kernels_compiled_for_sm103a_without_fast_math():
    from temporal_blocked_jacobi_gb300 import _build
    flags = " ".join(_build.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in flags
    assert "-fmad=false" in flags and "-ftz=false" in flags
    assert "use_fast_math" not in flags


def header_enum_values():
    """name -> value of every enumerator in include/jacobi.h."""
    text = open(os.path.join(ROOT, "include", "jacobi.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    values = {}
    for body in re.findall(r"typedef\s+enum\s*\{(.*?)\}", text, flags=re.S):
        nxt = 0
        for item in body.split(","):
            item = item.strip()
            if not item:
                continue
            m = re.match(r"(\w+)\s*(?:=\s*(-?\d+))?$", item)
            assert m, item
            nxt = int(m.group(2)) if m.group(2) is not None else nxt
            values[m.group(1)] = nxt
            nxt += 1
    return values


def test_binding_constants_match_the_header():
    from temporal_blocked_jacobi_gb300 import jacobi
    v = header_enum_values()
    assert v["JACOBI_SYNC"] == jacobi.SYNC
    assert v["JACOBI_EXACT_TEMPORAL_BLOCKED"] == jacobi.EXACT_TEMPORAL_BLOCKED
    assert v["JACOBI_BLOCK_ASYNC"] == jacobi.BLOCK_ASYNC
    assert v["JACOBI_CONTROL_HOST"] == jacobi.CONTROL_HOST
    assert v["JACOBI_CONTROL_DEVICE"] == jacobi.CONTROL_DEVICE
    assert v["JACOBI_CONTROL_PERSISTENT"] == jacobi.CONTROL_PERSISTENT
    assert jacobi.CONTROLS == {"host": 0, "device": 1, "persistent": 2}
    for name, val in (("JACOBI_OK", jacobi.OK),
                      ("JACOBI_ERR_INVALID_ARG", jacobi.ERR_INVALID_ARG),
                      ("JACOBI_ERR_CUDA", jacobi.ERR_CUDA),
                      ("JACOBI_ERR_NOT_CONVERGED", jacobi.ERR_NOT_CONVERGED),
                      ("JACOBI_ERR_NONFINITE", jacobi.ERR_NONFINITE),
                      ("JACOBI_ERR_UNSUPPORTED", jacobi.ERR_UNSUPPORTED)):
        assert v[name] == val, name
