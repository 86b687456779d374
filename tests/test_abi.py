"""The C-ABI library builds for sm_103a, loads, and exports every function
declared in include/*.h; argument validation and the planner run on the host
without a GPU."""
import ctypes
import os
import re

import pytest

import dense_fp32_sgemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^SGEMM_API\s+[^(]*?\b(sgemm_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    sg.build()
    return sg.library()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "sgemm_run" in names and "sgemm_run_host" in names
    assert len(names) == len(set(names))
    assert set(names) == set(sg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(sg.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_library_is_in_tree_and_built_for_sm_103a(lib):
    path = sg.library_path()
    assert path.startswith(ROOT)
    log = open(os.path.join(os.path.dirname(path), "ptxas.log")).read()
    assert "for 'sm_103a'" in log
    assert "bytes spill stores" in log
    # No kernel spills registers to local memory.
    spills = re.findall(r"(\d+) bytes spill stores", log)
    assert all(int(s) == 0 for s in spills), spills


def test_status_strings(lib):
    assert sg.status_string(0) == "SGEMM_OK"
    assert sg.status_string(5) == "SGEMM_ERR_DEVICE_TIMEOUT"
    assert sg.status_string(99) == "SGEMM_ERR_UNKNOWN"


@pytest.mark.parametrize("args", [
    dict(M=-1), dict(N=-2), dict(K=-3),
    dict(lda=3), dict(ldb=4), dict(ldc=4),
    dict(A=None), dict(B=None), dict(C=None),
    dict(A=4098), dict(C=8194),
])
def test_invalid_arguments_rejected_before_any_device_call(lib, args):
    call = dict(M=4, N=5, K=6, alpha=1.0, A=4096, lda=6, B=8192, ldb=5, beta=0.0,
                C=16384, ldc=5)
    call.update(args)
    st = sg.sgemm_run(call["M"], call["N"], call["K"], call["alpha"], call["A"], call["lda"],
                      call["B"], call["ldb"], call["beta"], call["C"], call["ldc"])
    assert st == 1, sg.status_string(st)


@pytest.mark.parametrize("args", [dict(M=-1), dict(lda=3), dict(A=None), dict(B=4098), dict(C=None)])
def test_3xtf32_arguments_rejected_before_any_device_call(lib, args):
    call = dict(M=4, N=5, K=6, alpha=1.0, A=4096, lda=6, B=8192, ldb=5, beta=0.0,
                C=16384, ldc=5)
    call.update(args)
    st = sg.sgemm_run_3xtf32(call["M"], call["N"], call["K"], call["alpha"], call["A"],
                             call["lda"], call["B"], call["ldb"], call["beta"], call["C"],
                             call["ldc"])
    assert st == 1, sg.status_string(st)
    assert sg.sgemm_run_3xtf32(0, 5, 6, 1.0, None, 6, None, 5, 0.0, None, 5) == 0


@pytest.mark.parametrize("bias,activation", [(None, 2), (None, -1), (4098, 0), (4097, 1)])
def test_epilogue_arguments_rejected_before_any_device_call(lib, bias, activation):
    st = sg.sgemm_run_epilogue(4, 5, 6, 1.0, 4096, 6, 8192, 5, 0.0, 16384, 5, bias, activation)
    assert st == 1, sg.status_string(st)
    st = sg.sgemm_run_3xtf32_epilogue(4, 5, 6, 1.0, 4096, 6, 8192, 5, 0.0, 16384, 5, bias,
                                      activation)
    assert st == 1, sg.status_string(st)


def test_empty_output_is_a_no_op_without_device(lib):
    assert sg.sgemm_run(0, 5, 6, 1.0, None, 6, None, 5, 0.0, None, 5) == 0
    assert sg.sgemm_run(4, 0, 6, 1.0, None, 6, None, 1, 0.0, None, 1) == 0


def test_alpha_zero_needs_no_operands(lib):
    # Validation accepts NULL A/B when alpha == 0; without a GPU the call then
    # stops at the device check.
    st = sg.sgemm_run(4, 5, 6, 0.0, None, 6, None, 5, 1.0, 4096, 5)
    assert st in (0, 6)


def test_probe_argument_checks(lib):
    assert lib.sgemm_probe_ffma(0, 0, 1, 4096, None) == 1
    assert lib.sgemm_probe_read(4100, 16, 4096, 1, None) == 1
    assert lib.sgemm_probe_read(4096, 6, 4096, 1, None) == 1
    assert lib.sgemm_probe_hold(0, None) == 1
    assert lib.sgemm_probe_hold(1000000001, None) == 1


def test_hooks_validate(lib):
    with pytest.raises(sg.SgemmError):
        sg.set_plan_override(sg.VARIANT_SMALL + 1, 0)
    with pytest.raises(sg.SgemmError):
        sg.set_tile_config(2, 4, 16)
    with pytest.raises(sg.SgemmError):
        sg.set_tile_config(3, 3, 12)
    with pytest.raises(sg.SgemmError):
        sg.set_tile_config(3, 3, 8)
    with pytest.raises(sg.SgemmError):
        sg.set_wait_timeout_ns(0, -5)
    for bk in (0, 8, 24, 64):
        with pytest.raises(sg.SgemmError):
            sg.set_3xtf32_config(bk, True)
    assert lib.sgemm_set_3xtf32_config(16, 2, 0, 0) == 1
    assert lib.sgemm_set_3xtf32_config(16, -2, 0, 0) == 1
    assert lib.sgemm_set_3xtf32_config(16, -1, -1, 0) == 1
    assert lib.sgemm_set_3xtf32_config(16, -1, 9, 0) == 1
    assert lib.sgemm_set_3xtf32_config(16, -1, 0, 3) == 1
    assert lib.sgemm_set_3xtf32_config(32, -1, 0, 2) == 1
    sg.set_3xtf32_config(32, False)
    sg.set_3xtf32_config(16, None)
    sg.set_plan_override(-1, 0)
    sg.set_tile_config(3, 3, 16)
    sg.set_wait_timeout_ns(0, -1)
