"""CPU-side checks of the C ABI: liblla.so builds, loads, exports every symbol
include/lla.h declares, and rejects bad arguments on the host before touching
the GPU. No call here reaches a kernel (every call fails validation first)."""
import ctypes
import os
import re

import pytest

from log_linear_attention_gb300 import binding, build, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lla_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"lla_forward", "lla_decode_step", "lla_forward_ws", "lla_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert binding.status_string(code).startswith("LLA_")
    assert binding.status_string(7) == "unknown lla status"


@pytest.mark.parametrize("T", [1, 2, 3, 64, 2048, 8192, 65536, 100000])
def test_num_levels(lib, T):
    assert binding.num_levels(T) == inputs.num_levels(T)


def test_workspace_size(lib):
    assert binding.workspace_size(1, 1, 64, 16, 16, 16, None) > 0
    assert binding.workspace_size(1, 1, 64, 16, 16, 48, None) == 0  # chunk not a power of two in range
    assert binding.workspace_size(1, 1, 65, 16, 16, 16, None) == 0  # T % chunk != 0
    assert binding.workspace_size(1, 1, 64, 256, 16, 16, None) == 0  # dk too large


A = 4096  # a 16-byte-aligned fake address: only ever used in calls that fail validation


def _fwd(lib, ptrs, B=1, H=1, T=64, dk=16, dv=16, chunk=16, dtype=1):
    q, k, v, a, lam, out = ptrs
    return lib.lla_forward(q, k, v, a, lam, out, B, H, T, dk, dv, chunk, None, dtype)


@pytest.mark.parametrize("case,expect", [
    (dict(ptrs=(None, A, A, A, A, A)), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A, A, A, A, A, None)), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A + 4, A, A, A, A, A)), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, chunk=48), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, chunk=8), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, T=72), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, B=0), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, dtype=5), binding.LLA_ERR_INVALID_ARG),
    (dict(ptrs=(A,) * 6, dk=200), binding.LLA_ERR_UNSUPPORTED),
])
def test_forward_rejects_bad_arguments(lib, case, expect):
    assert _fwd(lib, **case) == expect


def test_forward_ws_rejects_small_workspace(lib):
    st = lib.lla_forward_ws(A, A, A, A, A, A, 1, 1, 64, 16, 16, 16, None, 1, A, 16)
    assert st == binding.LLA_ERR_NOMEM


@pytest.mark.parametrize("args,expect", [
    (dict(dv=48), binding.LLA_ERR_UNSUPPORTED),
    (dict(dk=300), binding.LLA_ERR_UNSUPPORTED),
    (dict(Lmax=0), binding.LLA_ERR_INVALID_ARG),
    (dict(Lmax=41), binding.LLA_ERR_INVALID_ARG),
    (dict(t=None), binding.LLA_ERR_INVALID_ARG),
    (dict(t=A + 8), binding.LLA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments(lib, args, expect):
    a = dict(B=1, H=1, dk=16, dv=16, Lmax=5, dtype=1, t=A)
    a.update(args)
    st = lib.lla_decode_step(A, A, A, A, A, A, a["t"], A, None, a["B"], a["H"], a["dk"], a["dv"], a["Lmax"],
                             a["dtype"])
    assert st == expect


@pytest.mark.parametrize("args,expect", [
    (dict(dq=None), binding.LLA_ERR_INVALID_ARG),
    (dict(dlam=A + 4), binding.LLA_ERR_INVALID_ARG),
    (dict(dout=None), binding.LLA_ERR_INVALID_ARG),
    (dict(chunk=24), binding.LLA_ERR_INVALID_ARG),
    (dict(T=80, chunk=64), binding.LLA_ERR_INVALID_ARG),
    (dict(dv=129), binding.LLA_ERR_UNSUPPORTED),
])
def test_backward_rejects_bad_arguments(lib, args, expect):
    a = dict(dq=A, dlam=A, dout=A, T=64, dk=16, dv=16, chunk=16)
    a.update(args)
    st = lib.lla_backward(A, A, A, A, A, a["dout"], a["dq"], A, A, A, a["dlam"], 1, 1, a["T"], a["dk"], a["dv"],
                          a["chunk"], None, 1)
    assert st == expect


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "log_linear_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "lla_oracle" not in text, f
