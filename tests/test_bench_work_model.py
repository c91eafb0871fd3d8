"""The roofline denominators: the work model of one selection pass (FLOPs of the
leaf and scored intermediate levels, minimum bytes) at the benchmark's shapes,
recomputed by hand from the formula Hq*B*N*[g*K*C*2d + levels*g*K*g*2d] and
Q + K + 2 x pyramid + idx bytes, so that a change to the model is visible."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _shape(N, B=1, Hq=32, Hkv=2, K=8):
    return dict(B=B, N=N, Hq=Hq, Hkv=Hkv, K=K)


@pytest.mark.parametrize("N,scored,levels", [(32768, 6, 10), (65536, 7, 11), (131072, 8, 12), (262144, 9, 13)])
def test_flops_and_bytes_at_the_latency_shapes(N, scored, levels):
    a = bench.algorithmic(_shape(N))
    assert a["levels"] == levels
    # scored levels, the leaf level included: level l >= 2 is scored while M_l = N / (64 * 2^(l-1))
    # is above K = 8
    assert a["scored_intermediate_levels"] == scored - 1
    leaf = 32 * N * 16 * 64 * 128
    inter = 32 * N * (scored - 1) * 16 * 2 * 128
    assert a["leaf_flops"] == leaf and a["inter_flops"] == inter and a["flops"] == leaf + inter
    nodes = sum(bench.level_sizes(N))
    assert a["bytes"] == N * 32 * 64 * 2 + N * 2 * 64 * 2 + 2 * (2 * nodes * 64 * 4) + 2 * N * 8 * 4
    assert a["exps"] == 32 * N * (16 * 64 + (scored - 1) * 32)


def test_256k_figures():
    a = bench.algorithmic(_shape(262144))
    assert abs(a["flops"] - 1.3744e12) / 1.3744e12 < 1e-3
    assert abs(a["bytes"] - 1.166e9) / 1.166e9 < 1e-3
    assert a["leaf_row_gather_bytes"] == 2 * 262144 * 8 * 16 * 64 * 2


def test_no_scored_level_when_everything_fits_in_k():
    a = bench.algorithmic(_shape(512, K=8))  # 8 leaves: every level kept whole
    assert a["flops"] == 0 and a["scored_intermediate_levels"] == 0


def test_kernel_source_hash_ignores_comments_only():
    """The ncu traffic figure is tied to the kernel's code: a comment or blank-line
    edit keeps the hash, any code edit changes it."""
    src = "// header\n__global__ void k(int* a) {\n  /* block\n comment */ a[0] = 1;  // tail\n\n}\n"
    same = "__global__ void k(int* a) {\n  a[0] = 1;\n}\n// another note\n"
    other = "__global__ void k(int* a) {\n  a[0] = 2;\n}\n"
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(other)
    files = {"x.cu": src}
    bench.KERNEL_SOURCES["_probe"] = ["x.cu"]
    try:
        h1 = bench.source_sha1("_probe", read=files.get)
        files["x.cu"] = same
        h2 = bench.source_sha1("_probe", read=files.get)
        files["x.cu"] = other
        h3 = bench.source_sha1("_probe", read=files.get)
    finally:
        del bench.KERNEL_SOURCES["_probe"]
    assert h1 == h2 != h3
