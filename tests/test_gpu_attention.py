"""Stage-two block-sparse attention against the oracle, through the C ABI.

Tolerance: the probabilities enter the P.V product as bf16 (relative rounding
2^-9) while the softmax sum stays fp32, so each output element can be off by
about 2^-8 of the mean |v| it averages: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|."""
import numpy as np
import pytest
import torch

import oracle
import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _check(q, k, v, idx, t, causal):
    got = pisa.sparse_attention(q.to(DEV), k.to(DEV), v.to(DEV), idx.to(DEV), causal=causal).cpu().numpy()
    want = oracle.attention(q[:, t].float().numpy(), k.float().numpy(), v.float().numpy(),
                            idx[:, :, t].numpy(), t, causal=causal)
    np.testing.assert_allclose(got[:, t], want, rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("G,K,causal", [(16, 8, True), (4, 8, True), (1, 3, True), (8, 32, False), (2, 16, True)])
def test_random_blocks(G, K, causal):
    B, N, Hkv = 2, 700, 2
    q, k = synth.iid(B, N, G * Hkv, Hkv, seed=40 + G)
    _, v = synth.iid(B, N, G * Hkv, Hkv, seed=90 + G)
    idx = synth.random_blocks(B, Hkv, N, K, seed=5, causal=causal)
    _check(q, k, v, idx, np.arange(N), causal)


def test_every_block_selected_is_dense_attention():
    B, N, Hkv, G = 1, 300, 1, 16
    q, k = synth.iid(B, N, G, Hkv, seed=3)
    _, v = synth.iid(B, N, G, Hkv, seed=4)
    idx = torch.from_numpy(np.tile(np.arange(5, dtype=np.int32), (B, Hkv, N, 1)))
    _check(q, k, v, idx, np.arange(N), True)


def test_forward_on_the_selection():
    """Select with the pyramid, then attend over the selected blocks."""
    q, k, w = synth.make("tiny-2k")
    _, v = synth.iid(1, w["N"], w["Hq"], w["Hkv"], seed=77)
    pyr = pisa.build_pyramid(k.to(DEV))
    idx, _ = pisa.select_prefill(q.to(DEV), pyr, w["K"], with_scores=False)
    _check(q, k, v, idx.cpu(), np.arange(0, w["N"], 5), True)


def test_forward_at_full_size_sampled():
    """Stage two at the benchmark's own size (256K tokens, the pass's selection, the
    launch configuration the benchmark times), checked at a seeded sample of positions
    plus the last 64."""
    q, k, w = synth.make("latency-256k")
    _, v = synth.iid(1, w["N"], w["Hq"], w["Hkv"], seed=77)
    qd, kd = q.to(DEV), k.to(DEV)
    pyr = pisa.build_pyramid(kd)
    idx, _ = pisa.select_prefill(qd, pyr, w["K"], with_scores=False)
    got = pisa.sparse_attention(qd, kd, v.to(DEV), idx, causal=True)
    rng = np.random.default_rng(7)
    N = w["N"]
    t = np.unique(np.concatenate([rng.choice(N - 64, 2048, replace=False), np.arange(N - 64, N)]))
    tt = torch.from_numpy(t).to(DEV)
    got_t = got[:, tt].cpu().numpy()
    idx_t = idx[:, :, tt].cpu().numpy()
    del got
    want = oracle.attention(q[:, t].float().numpy(), k.float().numpy(), v.float().numpy(), idx_t, t, causal=True)
    np.testing.assert_allclose(got_t, want, rtol=1e-2, atol=1e-2)
