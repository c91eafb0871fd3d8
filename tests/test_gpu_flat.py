"""The flat selector (every eligible leaf scored exactly) against the oracle's
flat selection, through the C ABI."""
import numpy as np
import pytest
import torch

import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

from parity import compare_flat, record

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _f32(x):
    return x.float().cpu().numpy()


def _run_flat(q, k, K, causal=True):
    qd, kd = q.to(DEV), k.to(DEV)
    pyr = pisa.Pyramid.allocate(kd)
    B, N, Hq, _ = q.shape
    ws = torch.empty(pisa.flat_workspace_bytes(B, N, Hq, k.shape[2], K), dtype=torch.uint8, device=DEV)
    idx, sc = pisa.select_flat(qd, pyr, K, causal=causal, workspace=ws)
    assert pisa.check_device_status(ws) == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


def _ok(st):
    assert st["unexcused"] == 0, st["messages"]
    assert st.get("score_bad", 0) == 0, st["messages"]
    assert st["excused"] <= 0.01 * st["rows"] + 2, st


def test_flat_tiny_all_queries():
    q, k, w = synth.make("tiny-2k")
    idx, sc = _run_flat(q, k, w["K"])
    st = compare_flat(idx, sc, _f32(q), _f32(k), np.arange(w["N"]), w["K"])
    record("flat tiny-2k", st)
    _ok(st)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("K", [1, 8, 32])
def test_flat_small_shapes(causal, K):
    q, k = synth.iid(2, 1000, 8, 2, seed=17)
    idx, sc = _run_flat(q, k, K, causal=causal)
    st = compare_flat(idx, sc, _f32(q), _f32(k), np.arange(1000), K, causal=causal)
    _ok(st)


def test_flat_latency_32k_sampled():
    q, k, w = synth.make("latency-32k")
    idx, sc = _run_flat(q, k, w["K"])
    N = w["N"]
    rng = np.random.default_rng(7)
    t = np.unique(np.concatenate([rng.choice(N - 256, 1024, replace=False), np.arange(N - 256, N)]))
    st = compare_flat(idx[:, :, t], sc[:, :, t], _f32(q[:, t]), _f32(k), t, w["K"])
    record("flat latency-32k (sampled)", st)
    _ok(st)


def test_flat_latency_256k_sampled():
    """The flat selector at the largest benchmark size (4096 leaves per query), sampled."""
    q, k, w = synth.make("latency-256k")
    idx, sc = _run_flat(q, k, w["K"])
    N = w["N"]
    rng = np.random.default_rng(11)
    t = np.unique(np.concatenate([rng.choice(N - 64, 512, replace=False), np.arange(N - 64, N)]))
    st = compare_flat(idx[:, :, t], sc[:, :, t], _f32(q[:, t]), _f32(k), t, w["K"])
    record("flat latency-256k (sampled)", st)
    _ok(st)


def test_flat_equals_pyramid_when_every_leaf_reaches_the_leaf_level():
    """M_2 <= K: the walk scores every eligible leaf, exactly like the flat selector."""
    q, k = synth.iid(1, 2048, 32, 2, seed=23)  # M_2 = 16
    fi, fs = _run_flat(q, k, 16)
    kd = k.to(DEV)
    pyr = pisa.build_pyramid(kd)
    pi, ps = pisa.select_prefill(q.to(DEV), pyr, 16)
    np.testing.assert_array_equal(fi, pi.cpu().numpy())
    # same leaf kernel; a warp sums a chunk on its packed path only when both of its
    # queries see the whole chunk, so the two tilings can differ in the last bits
    np.testing.assert_allclose(fs, ps.cpu().numpy(), rtol=1e-6, atol=0)
