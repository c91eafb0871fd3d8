"""The debug build (-DPISA_DEBUG_BOUNDS) range-checks every gathered index on the device
(a failed check records PISA_ERR_DEVICE_BOUNDS and the access is replaced by a harmless
one).  On the parity workloads no check fails and the indices are those of the default
build, bit for bit.  The debug library runs in a child process so that this process
keeps the default one."""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import build, synth
sys.path.insert(0, sys.argv[1] + "/tests")
from test_gpu_debug_bounds import run_cases
pisa.load(build.build(extra_flags=["-DPISA_DEBUG_BOUNDS"], name="libpisa_debug"))
res = run_cases()
np.savez(sys.argv[2], **res)
"""


def run_cases():
    """Prefill at G = 4 (K = 8), G = 16 (K = 8) and G = 16 (K = 32, ragged), and decode
    steps; returns the indices and every call's status word."""
    out = {}
    cases = [("tiny", synth.make("tiny-2k")[:2], 8), ("g16", synth.iid(1, 20000, 32, 2, seed=4), 8),
             ("ragged", synth.make("ragged-16421")[:2], 32)]
    for name, (q, k), K in cases:
        B, N, Hq, _ = q.shape
        pyr = pisa.build_pyramid(k.cuda())
        ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, k.shape[2], K), dtype=torch.uint8, device="cuda")
        idx, _ = pisa.select_prefill(q.cuda(), pyr, K, workspace=ws, with_scores=False)
        torch.cuda.synchronize()
        out[name] = idx.cpu().numpy()
        out[name + "_status"] = np.array(pisa.check_device_status(ws))
    B, Hq, Hkv, K = 4, 32, 2, 8
    cache, g = synth.decode_context(B, 5000, 5100, Hkv, seed=2)
    pyr = pisa.Pyramid.allocate(cache.cuda(), with_lengths=True)
    pisa.build_pyramid(pyr, N=5000)
    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device="cuda")
    steps = []
    for _ in range(6):
        qn, kn = synth.decode_step(g, B, Hq, Hkv)
        idx, _ = pisa.decode_append_and_select(qn.cuda(), kn.cuda(), pyr, K, workspace=ws)
        steps.append(idx.cpu().numpy())
    torch.cuda.synchronize()
    out["decode"] = np.stack(steps)
    out["decode_status"] = np.array(pisa.check_device_status(ws))
    return out


def test_debug_build_checks_pass_and_match_the_default_build():
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "debug.npz")
        r = subprocess.run([sys.executable, "-c", CHILD, ROOT, path], capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, r.stderr[-3000:]
        dbg = dict(np.load(path))
    ref = run_cases()
    for name in ("tiny", "g16", "ragged", "decode"):
        assert int(dbg[name + "_status"]) == 0, (name, int(dbg[name + "_status"]))
        assert int(ref[name + "_status"]) == 0
        assert np.array_equal(dbg[name], ref[name]), name
