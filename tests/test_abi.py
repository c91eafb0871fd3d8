"""The C ABI library loads, exports every function include/pisa.h declares, and
its host-only logic (level geometry, workspace sizing, argument checks) works
without a GPU.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import oracle
import pyramid_top_block_gb300 as pisa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pisa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pisa_\w+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = pisa.load()
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 200, 2048, 16421, 131073, 262144, 1 << 30])
def test_level_geometry_matches_oracle(n):
    assert pisa.num_levels(n) == oracle.num_levels(n)
    assert pisa.pyramid_nodes(n) == oracle.total_nodes(n)
    sizes = oracle.level_sizes(n)
    off = 0
    for lvl, m in enumerate(sizes, start=1):
        assert pisa.level_offset(n, lvl) == off
        off += m


def test_workspace_sizes():
    ws = pisa.select_workspace_bytes(1, 262144, 32, 2, 8)
    assert ws >= 4 * 262144 * 2 * 8
    assert pisa.select_workspace_bytes(1, 100, 32, 2, 33) == 0      # K too large
    assert pisa.select_workspace_bytes(1, 100, 24, 2, 8) == 0       # group of 12
    assert pisa.select_workspace_bytes(1, 100, 30, 4, 8) == 0       # Hq % Hkv != 0
    assert pisa.decode_workspace_bytes(16, 32, 2, 8) >= 4


def test_argument_errors_without_launch():
    lib = pisa.load()
    assert lib.pisa_build_pyramid(None, 10, None) == 1
    st = pisa._PyrStruct(0x1000, 0x2000, None, 1, 2, 32, 64, 2, 128)   # d = 32
    assert lib.pisa_build_pyramid(ctypes.byref(st), 10, None) == 2
    st = pisa._PyrStruct(0x1000, 0x2000, None, 1, 2, 64, 64, 2, 128)
    assert lib.pisa_build_pyramid(ctypes.byref(st), 129, None) == 1      # N > n_cap
    assert lib.pisa_build_pyramid(ctypes.byref(st), 0, None) == 1
    # select: NULL outputs, bad K, bad group, small workspace
    assert lib.pisa_select_prefill(ctypes.c_void_p(0x3000), 32, ctypes.byref(st), 128, 8, 1,
                                   None, None, ctypes.c_void_p(0x4000), 1 << 20, None) == 1
    assert lib.pisa_select_prefill(ctypes.c_void_p(0x3000), 32, ctypes.byref(st), 128, 40, 1,
                                   ctypes.c_void_p(0x5000), None, ctypes.c_void_p(0x4000), 1 << 20, None) == 2
    assert lib.pisa_select_prefill(ctypes.c_void_p(0x3000), 6, ctypes.byref(st), 128, 8, 1,
                                   ctypes.c_void_p(0x5000), None, ctypes.c_void_p(0x4000), 1 << 20, None) == 2
    assert lib.pisa_select_prefill(ctypes.c_void_p(0x3000), 32, ctypes.byref(st), 128, 8, 1,
                                   ctypes.c_void_p(0x5000), None, ctypes.c_void_p(0x4000), 16, None) == 3
    # decode needs lengths
    assert lib.pisa_decode_append_and_select(ctypes.c_void_p(0x3000), ctypes.c_void_p(0x3000), 32,
                                             ctypes.byref(st), 8, ctypes.c_void_p(0x5000), None,
                                             ctypes.c_void_p(0x4000), 1 << 20, None) == 1


def test_status_strings():
    for s in range(7):
        assert pisa.status_string(s)
    assert pisa.status_string(99) == "unknown status"
