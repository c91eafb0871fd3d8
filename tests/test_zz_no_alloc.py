"""The allocation-free prefill entry point (pisa_select_prefill_noalloc).

It serves callers that cannot allocate device memory themselves (a host
framework that owns all device memory and passes only input and output
buffers, or a request path where cudaMalloc is not allowed).  It must give
the same selection as pisa_select_prefill with a caller workspace, call after
call, although its built-in scratch keeps the previous call's contents.

This file is collected last on purpose, and also passes when run alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

from parity import REL

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _call_noalloc(lib, qd, pyr, K, causal, idx, sc):
    st = pyr.struct()
    return lib.pisa_select_prefill_noalloc(ctypes.c_void_p(qd.data_ptr()), qd.shape[2], ctypes.byref(st),
                                           qd.shape[1], K, int(causal), ctypes.c_void_p(idx.data_ptr()),
                                           ctypes.c_void_p(sc.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _problem(seed, N, Hq, Hkv):
    q, k = synth.iid(1, N, Hq, Hkv, seed=seed)
    qd, kd = q.to(DEV), k.to(DEV)
    return qd, pisa.build_pyramid(kd)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    lib = pisa.load()
    # two different problems in a row: the second call must not see the first's leftovers
    cases = [(41, 8192, 32, 2, 8, True), (42, 5000, 16, 4, 5, False)]
    for seed, N, Hq, Hkv, K, causal in cases:
        qd, pyr = _problem(seed, N, Hq, Hkv)
        ref_idx, ref_sc = pisa.select_prefill(qd, pyr, K, causal=causal)
        idx = torch.full((1, Hkv, N, K), -7, dtype=torch.int32, device=DEV)
        sc = torch.full((1, Hkv, N, K), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_noalloc(lib, qd, pyr, K, causal, idx, sc) == 0
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        a, b = sc.cpu().numpy(), ref_sc.cpu().numpy()
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin)
        assert np.all(a[~fin] == b[~fin])
        assert np.all(np.abs(a[fin] - b[fin]) <= REL * np.maximum(1.0, np.abs(b[fin])))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = pisa.load()
    limit = 32 << 20
    N = 1 << 22  # 4M tokens: the workspace these sizes need is far above 32 MiB
    assert pisa.select_workspace_bytes(1, N, 32, 2, 8) > limit
    kd = torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16, device=DEV)
    pyr = pisa.Pyramid.allocate(kd)
    st = pyr.struct()
    st.n_cap = N  # never dereferenced: the size check fails before any launch
    rc = lib.pisa_select_prefill_noalloc(ctypes.c_void_p(kd.data_ptr()), 32, ctypes.byref(st), N, 8, 1,
                                         ctypes.c_void_p(kd.data_ptr()), None, None)
    assert rc == 3


def test_noalloc_status_word_reads_a_device_side_timeout():
    """A kernel-side error of this entry point lands in its built-in scratch, where
    the caller has no workspace to read it from: pisa_noalloc_device_status reads
    it.  The timeout is planted by the bounded-wait self-test, run on the scratch
    itself (nothing faults); the next selection clears it."""
    lib = pisa.load()
    addr = pisa.noalloc_prepare()
    assert addr != 0 and addr % 256 == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.pisa_selftest_bounded_wait(ctypes.c_void_p(addr), 256, 0, stream) == 0
    assert pisa.noalloc_device_status() == 5  # PISA_ERR_DEVICE_TIMEOUT
    qd, pyr = _problem(43, 3000, 32, 2)
    idx, _ = pisa.select_prefill_noalloc(qd, pyr, 8, with_scores=False)
    assert pisa.noalloc_device_status() == 0
    ref, _ = pisa.select_prefill(qd, pyr, 8, with_scores=False)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref)
