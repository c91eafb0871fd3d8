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


def test_debug_bounds_build_compiles_and_exports_the_same_functions():
    """The -DPISA_DEBUG_BOUNDS variant (device-side index checks) builds beside the default
    library and exports the same C ABI; nothing is launched."""
    from pyramid_top_block_gb300 import build
    path = build.build(extra_flags=["-DPISA_DEBUG_BOUNDS"], name="libpisa_debug")
    assert os.path.basename(path) == "libpisa_debug.so" and path != build.LIB
    lib = ctypes.CDLL(path)
    for n in _declared():
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
    # entries (b, kv, t, slot) are indexed in 32 bits with room for a block past the end
    assert pisa.select_workspace_bytes(1, (1 << 26) - 31, 16, 1, 32) == 0   # 2^31 - 992 entries
    assert pisa.select_workspace_bytes(1, (1 << 26) - 32769, 16, 1, 32) > 0  # just below 2^31 - 2^20
    assert pisa.decode_workspace_bytes(16, 32, 2, 8) >= 4


def test_argument_errors_without_launch():
    lib = pisa.load()
    assert lib.pisa_build_pyramid(None, 10, None) == 1
    st = pisa._PyrStruct(0x1000, 0x2000, None, 1, 2, 32, 64, 2, 128)   # d = 32
    assert lib.pisa_build_pyramid(ctypes.byref(st), 10, None) == 2
    st = pisa._PyrStruct(0x1000, 0x2000, None, 40000, 2, 64, 64, 2, 128)  # B * Hkv > 65535
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


def test_host_selection_argument_errors_without_launch():
    """pisa_select_prefill_host rejects bad arguments before it touches a stream."""
    lib = pisa.load()
    st = pisa._PyrStruct(0x1000, 0x2000, 0x6000, 1, 2, 64, 64, 2, 128)
    vp = ctypes.c_void_p
    good = dict(K_host=vp(0x7000), Q_host=vp(0x8000), Q_dev=vp(0x3000), idx_host=vp(0x9000), idx_dev=vp(0x5000))

    def call(N=128, Hq=32, K=8, ws_bytes=1 << 30, **over):
        a = dict(good, **over)
        return lib.pisa_select_prefill_host(ctypes.byref(st), a["K_host"], N, a["Q_host"], a["Q_dev"], Hq, K, 1,
                                            a["idx_host"], a["idx_dev"], vp(0x4000), ws_bytes, None, None)

    assert call(K_host=None) == 1
    assert call(Q_host=None) == 1
    assert call(idx_host=None) == 1
    assert call(idx_dev=None) == 1
    assert call(Q_dev=vp(0x3008)) == 1           # device Q not 16-byte aligned
    assert call(N=129) == 1                     # N > n_cap
    assert call(K=40) == 2                      # K too large
    assert call(Hq=6) == 2                      # group of 3
    assert call(ws_bytes=16) == 3               # workspace too small


def test_decode_workspace_counts_one_arrival_slot_per_sequence():
    assert pisa.decode_workspace_bytes(1, 32, 2, 8) >= 256 + 4
    assert pisa.decode_workspace_bytes(300, 32, 2, 8) >= 256 + 4 * 300


def test_bounded_wait_selftest_argument_errors_without_launch():
    lib = pisa.load()
    vp = ctypes.c_void_p
    assert lib.pisa_selftest_bounded_wait(None, 256, 1000, None) == 1
    assert lib.pisa_selftest_bounded_wait(vp(0x4010), 256, 1000, None) == 1     # not 256-byte aligned
    assert lib.pisa_selftest_bounded_wait(vp(0x4000), 16, 1000, None) == 3      # workspace too small
    assert lib.pisa_selftest_bounded_wait(vp(0x4000), 256, -1, None) == 1
    assert lib.pisa_selftest_bounded_wait(vp(0x4000), 256, 1 << 40, None) == 1  # more than about 2 s


def test_status_strings():
    for s in range(7):
        assert pisa.status_string(s)
    assert pisa.status_string(99) == "unknown status"


def test_noalloc_argument_checks_match_the_workspace_entry_point():
    """The allocation-free entry point returns the codes pisa_select_prefill returns
    for the same arguments (same checks, same order) before its own size limit;
    nothing here reaches a CUDA call."""
    lib = pisa.load()
    vp = ctypes.c_void_p
    st = pisa._PyrStruct(0x1000, 0x2000, None, 1, 2, 64, 64, 2, 128)
    big = pisa._PyrStruct(0x1000, 0x2000, None, 1, 2, 64, 64, 2, 1 << 22)

    def both(pyr, Hq, N, K, idx=vp(0x5000), Q=vp(0x3000)):
        a = lib.pisa_select_prefill(Q, Hq, ctypes.byref(pyr), N, K, 1, idx, None, vp(0x4000), 1 << 40, None)
        b = lib.pisa_select_prefill_noalloc(Q, Hq, ctypes.byref(pyr), N, K, 1, idx, None, None)
        return a, b

    assert both(st, 32, 128, 33) == (2, 2)                 # K above 32: unsupported
    assert both(st, 24, 128, 8) == (2, 2)                  # group of 12
    assert both(st, 32, 129, 8) == (1, 1)                  # N > n_cap
    assert both(st, 32, 128, 8, idx=None) == (1, 1)        # no output
    assert both(st, 32, 128, 8, Q=vp(0x3008)) == (1, 1)    # Q not 16-byte aligned
    assert lib.pisa_select_prefill_noalloc(vp(0x3000), 32, None, 128, 8, 1, vp(0x5000), None, None) == 1
    # valid arguments beyond the scratch: only the no-allocation entry point refuses
    assert lib.pisa_select_prefill_noalloc(vp(0x3000), 32, ctypes.byref(big), 1 << 22, 8, 1, vp(0x5000), None,
                                           None) == 3
