"""Host-buffer selection (pisa_select_prefill_host): keys and queries copied in by
query runs on a copy stream while the selection runs, indices copied back per run.
Its results must be those of the device-resident build + selection, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

from parity import compare_prefill

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _device_reference(q, k, K, causal):
    pyr = pisa.build_pyramid(k.to(DEV))
    idx, _ = pisa.select_prefill(q.to(DEV), pyr, K, causal=causal, with_scores=False)
    torch.cuda.synchronize()
    return idx.cpu()


@pytest.mark.parametrize("B,N,Hq,Hkv,K,causal", [
    (1, 40000, 32, 2, 8, True),    # three query chunks of 2^14 tokens, ragged last
    (2, 33000, 16, 2, 8, False),   # two batches, non-causal, ragged last chunk
    (1, 20000, 8, 1, 16, True),    # K > 8 (generic walk), one KV head
])
def test_host_path_matches_device_path(B, N, Hq, Hkv, K, causal):
    q, k = synth.iid(B, N, Hq, Hkv, seed=11)
    want = _device_reference(q, k, K, causal)
    pyr = pisa.Pyramid.allocate(torch.empty(B, N, Hkv, 64, dtype=torch.bfloat16, device=DEV), with_lengths=True)
    qh, kh = q.pin_memory(), k.pin_memory()
    idx_h = pisa.select_prefill_host(qh, kh, pyr, K, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(idx_h, want)
    assert pyr.lengths.cpu().tolist() == [N] * B
    assert torch.equal(pyr.keys.cpu(), k)


def test_host_path_into_a_larger_pyramid_and_repeated_calls():
    """n_cap > N: the keys land in the first N rows of each sequence (pitched copy);
    back-to-back calls on the same buffers give the same bits."""
    B, N, n_cap, Hq, Hkv, K = 2, 17000, 20000, 16, 2, 8
    q, k = synth.iid(B, N, Hq, Hkv, seed=12)
    want = _device_reference(q, k, K, True)
    pyr = pisa.Pyramid.allocate(torch.zeros(B, n_cap, Hkv, 64, dtype=torch.bfloat16, device=DEV), with_lengths=True)
    qh, kh = q.pin_memory(), k.pin_memory()
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, Hkv, K), dtype=torch.uint8, device=DEV)
    qd = torch.empty(B, N, Hq, 64, dtype=torch.bfloat16, device=DEV)
    idd = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(3):
        idx_h = torch.full((B, Hkv, N, K), -7, dtype=torch.int32).pin_memory()
        pisa.select_prefill_host(qh, kh, pyr, K, idx_host=idx_h, q_dev=qd, idx_dev=idd, workspace=ws)
        outs.append(idx_h)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, want)
    assert torch.equal(pyr.keys[:, :N].cpu(), k)


def test_host_path_sampled_rows_match_the_oracle():
    B, N, Hq, Hkv, K = 1, 40000, 32, 2, 8
    q, k = synth.iid(B, N, Hq, Hkv, seed=13)
    pyr = pisa.Pyramid.allocate(torch.empty(B, N, Hkv, 64, dtype=torch.bfloat16, device=DEV), with_lengths=True)
    idx_h = pisa.select_prefill_host(q.pin_memory(), k.pin_memory(), pyr, K)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 64), np.linspace(64, N - 1, 40).astype(np.int64),
                                     [16383, 16384, 32767, 32768, N - 1]]))
    st = compare_prefill(idx_h[:, :, rows].numpy(), None, q[:, rows].float().numpy(), k.float().numpy(), rows, K,
                         True)
    assert st["unexcused"] == 0, st["messages"]
