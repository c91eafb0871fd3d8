"""PISA-1 / PISA-2 score modes (mean, and mean + half the variance of the child
logits; raw-key logits at the leaf) of the prefill walk and of the flat
selector against the oracle's modes, through the C ABI."""
import numpy as np
import pytest
import torch

import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

from parity import compare_flat, compare_prefill, record

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _f32(x):
    return x.float().cpu().numpy()


def _ok(st):
    assert st["unexcused"] == 0, st["messages"]
    assert st.get("score_bad", 0) == 0, st["messages"]
    assert st["excused"] <= 0.01 * st["rows"] + 2, st


def _prefill(q, k, K, mode, causal=True):
    pyr = pisa.build_pyramid(k.to(DEV))
    B, N, Hq, _ = q.shape
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, k.shape[2], K), dtype=torch.uint8, device=DEV)
    idx, sc = pisa.select_prefill(q.to(DEV), pyr, K, causal=causal, workspace=ws, mode=mode)
    assert pisa.check_device_status(ws) == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("K,causal", [(8, True), (8, False), (3, True), (16, True), (32, False)])
def test_prefill_modes_small(mode, K, causal):
    q, k = synth.iid(2, 3000, 32, 2, seed=31)
    idx, sc = _prefill(q, k, K, mode, causal)
    st = compare_prefill(idx, sc, _f32(q), _f32(k), np.arange(3000), K, causal=causal, mode=mode)
    _ok(st)


@pytest.mark.parametrize("mode", [1, 2])
def test_prefill_modes_ragged_structured(mode):
    q, k, w = synth.make("ragged-16421")
    idx, sc = _prefill(q, k, w["K"], mode)
    t = np.arange(0, w["N"], 3)
    st = compare_prefill(idx[:, :, t], sc[:, :, t], _f32(q[:, t]), _f32(k), t, w["K"], mode=mode)
    record(f"ragged-16421 mode {mode}", st)
    _ok(st)


@pytest.mark.parametrize("mode", [1, 2])
def test_prefill_modes_at_256k_sampled(mode):
    """The score modes at the benchmark's largest size (the launch configuration the
    benchmark times for them), compared at a seeded sample of positions plus the last 1024."""
    q, k, w = synth.make("latency-256k")
    idx, sc = _prefill(q, k, w["K"], mode)
    N = w["N"]
    rng = np.random.default_rng(3 + mode)
    t = np.unique(np.concatenate([rng.choice(N - 1024, 8192, replace=False), np.arange(N - 1024, N)]))
    st = compare_prefill(idx[:, :, t], sc[:, :, t], _f32(q[:, t]), _f32(k), t, w["K"], mode=mode)
    record(f"latency-256k mode {mode} (sampled)", st)
    _ok(st)


@pytest.mark.parametrize("mode", [1, 2])
def test_flat_modes(mode):
    q, k = synth.iid(1, 2000, 16, 1, seed=37)
    pyr = pisa.Pyramid.allocate(k.to(DEV))
    idx, sc = pisa.select_flat(q.to(DEV), pyr, 8, mode=mode)
    st = compare_flat(idx.cpu().numpy(), sc.cpu().numpy(), _f32(q), _f32(k), np.arange(2000), 8, mode=mode)
    _ok(st)


def test_unknown_mode_is_rejected():
    q, k = synth.iid(1, 128, 4, 1, seed=1)
    pyr = pisa.build_pyramid(k.to(DEV))
    with pytest.raises(pisa.PisaError):
        pisa.select_prefill(q.to(DEV), pyr, 2, mode=3)
