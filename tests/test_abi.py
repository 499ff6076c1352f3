"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
function include/based.h declares, rejects bad arguments before touching a device, and the work
partition covers every chunk once with correct prefix slots."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from linear_attention_gb300 import build as lbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "based.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"BASED_API\s+[\w\s\*]+?\b(based_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    lbuild.build()
    from linear_attention_gb300 import based
    return based.library()


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("based_fwd", "based_fwd_ws", "based_fwd_workspace_size", "based_fwd_host",
              "based_fwd_strerror", "based_strerror", "based_device_status",
              "based_selftest_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (based_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_strerror_names_every_code(lib):
    for code in range(0, -13, -1):
        name = lib.based_fwd_strerror(code).decode()
        assert name != "unknown error code"
        assert lib.based_strerror(code).decode() == name  # the older name is the same function
    assert lib.based_fwd_strerror(-99).decode() == "unknown error code"
    assert lib.based_strerror(-99).decode() == "unknown error code"
    assert lib.based_abi_version() == 10100


def _call(lib, q=16, k=16, v=16, B=1, T=8, H=1, K=16, V=64, o=4096):
    # fake but aligned "device" addresses: argument checks run before any CUDA call
    return lib.based_fwd(q, k, v, B, T, H, K, V, ctypes.c_float(-1.0), o, None)


def test_argument_errors_are_reported_before_launch(lib):
    base = 1 << 40
    ok = dict(q=base, k=base + (1 << 20), v=base + (2 << 20), o=base + (3 << 20))
    assert _call(lib, **{**ok, "q": 0}) == -1
    assert _call(lib, **{**ok, "o": 0}) == -1
    assert _call(lib, **ok, K=4) == -2
    assert _call(lib, **ok, K=32) == -2
    assert _call(lib, **ok, V=96) == -3
    assert _call(lib, **ok, T=0) == -4
    assert _call(lib, **ok, B=-1) == -4
    assert _call(lib, **ok, B=1 << 16, T=1 << 16, H=1) == -4
    assert _call(lib, **{**ok, "v": base + (2 << 20) + 8}) == -5
    assert _call(lib, **{**ok, "o": ok["v"] + 64}) == -6
    assert _call(lib, **{**ok, "o": ok["q"]}) == -6


def test_bf16_output_argument_errors(lib):
    # same checks on the bf16-output entry point; its output spans B*T*H*V*2 bytes
    def call(q, k, v, o, B=1, T=8, H=1, K=16, V=64):
        return lib.based_fwd_bf16_out(q, k, v, B, T, H, K, V, ctypes.c_float(-1.0), o, None, 0,
                                      None, None, None)
    base = 1 << 40
    q, k, v = base, base + (1 << 20), base + (2 << 20)
    assert call(q, k, v, 0) == -1
    assert call(q, k, v, base + (3 << 20), K=12) == -2
    assert call(q, k, v, base + (3 << 20), V=32) == -3
    assert call(q, k, v, base + (3 << 20) + 2) == -5
    assert call(q, k, v, v + 64) == -6
    # a bf16 output of 8 rows x 64 spans 1024 bytes: one that starts 1008 bytes before q
    # overlaps it
    assert call(q, k, v, q - 1008) == -6


def test_partition_and_prefix_slots():
    exe = os.path.join(tempfile.mkdtemp(), "partition_check")
    subprocess.run([lbuild.nvcc(), "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                    os.path.join(ROOT, "tests", "partition_check.cu")], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok")
