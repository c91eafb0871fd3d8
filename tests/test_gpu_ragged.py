"""Ragged batches (sequences of different lengths) and decode steps replayed from
a CUDA graph, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

from parity import compare_decode, pyramid_tolerance

pytestmark = pytest.mark.gpu

DEV = "cuda"
LENGTHS = [4000, 1, 130, 2049, 0]


def _ragged_cache(n_cap=4200, Hkv=2, seed=8):
    g = torch.Generator().manual_seed(seed)
    cache = torch.zeros(len(LENGTHS), n_cap, Hkv, 64, dtype=torch.bfloat16)
    for b, n in enumerate(LENGTHS):
        cache[b, :n] = torch.randn(n, Hkv, 64, generator=g).to(torch.bfloat16)
    return cache, g


def _valid_nodes_equal(got, cache, lengths):
    """Every node of sequence b's own levels matches the oracle's mean pyramid over
    lengths[b] tokens within the fp32 summation bound (GPU layout offsets come from
    n_cap, the oracle's from n)."""
    n_cap = cache.shape[1]
    for b, n in enumerate(lengths):
        if n == 0:
            continue
        kb = cache[b:b + 1].float().numpy()
        want = oracle.build_pyramid(kb, n=n)[0]
        tol = pyramid_tolerance(kb, n=n)[0]
        off_o = 0
        for lvl, m in enumerate(oracle.level_sizes(n), start=1):
            off_g = pisa.level_offset(n_cap, lvl)
            g = got[b, :, off_g:off_g + m].double().cpu().numpy()
            err = np.abs(g - want[:, off_o:off_o + m])
            assert (err <= tol[:, off_o:off_o + m]).all(), (b, lvl)
            off_o += m


def test_ragged_build_matches_oracle_per_sequence():
    cache, _ = _ragged_cache()
    pyr = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    pyr.lengths.copy_(torch.tensor(LENGTHS, dtype=torch.int32))
    pisa.build_pyramid_ragged(pyr)
    torch.cuda.synchronize()
    _valid_nodes_equal(pyr.summaries, cache, LENGTHS)


def test_ragged_build_with_equal_lengths_is_the_uniform_build():
    _, k = synth.iid(3, 2100, 8, 2, seed=2)
    a = pisa.Pyramid.allocate(k.to(DEV), with_lengths=True)
    a.lengths.fill_(2100)
    pisa.build_pyramid_ragged(a)
    b = pisa.build_pyramid(k.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(a.summaries, b.summaries)


def test_ragged_decode_matches_oracle_and_rebuild():
    Hq, Hkv, K, steps = 32, 2, 8, 40
    cache, g = _ragged_cache()
    B = cache.shape[0]
    pyr = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    pyr.lengths.copy_(torch.tensor(LENGTHS, dtype=torch.int32))
    pisa.build_pyramid_ragged(pyr)
    for s in range(steps):
        qn, kn = synth.decode_step(g, B, Hq, Hkv)
        idx, sc = pisa.decode_append_and_select(qn.to(DEV), kn.to(DEV), pyr, K)
        for b, n in enumerate(LENGTHS):
            cache[b, n + s] = kn[b]
        if s % 9 == 0 or s == steps - 1:
            torch.cuda.synchronize()
            lengths = np.array(LENGTHS) + s + 1
            st = compare_decode(idx.cpu().numpy(), sc.cpu().numpy(), qn.float().numpy(), cache.float().numpy(),
                                lengths, K)
            assert st["unexcused"] == 0 and st["score_bad"] == 0, st["messages"]
    torch.cuda.synchronize()
    final = [n + steps for n in LENGTHS]
    assert pyr.lengths.cpu().tolist() == final
    fresh = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    fresh.lengths.copy_(torch.tensor(final, dtype=torch.int32))
    pisa.build_pyramid_ragged(fresh)
    torch.cuda.synchronize()
    for b, n in enumerate(final):  # the incrementally kept pyramid equals a rebuild, bit for bit
        for lvl, m in enumerate(oracle.level_sizes(n), start=1):
            off = pisa.level_offset(cache.shape[1], lvl)
            assert torch.equal(pyr.summaries[b, :, off:off + m], fresh.summaries[b, :, off:off + m]), (b, lvl)


def test_decode_steps_replay_from_a_cuda_graph():
    """The decode step reads lengths on the device only, so a run of steps can be
    captured once and replayed; the replay gives the eager run's bits."""
    Hq, Hkv, K, steps = 16, 2, 8, 12
    cache, g = _ragged_cache(Hkv=Hkv)
    B = cache.shape[0]
    qs, ks = zip(*[synth.decode_step(g, B, Hq, Hkv) for _ in range(steps)])
    qd, kd = torch.stack(qs).to(DEV), torch.stack(ks).to(DEV)

    def fresh_state():
        p = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
        p.summaries.zero_()  # nodes past a sequence's own levels are never written: start both equal
        p.lengths.copy_(torch.tensor(LENGTHS, dtype=torch.int32))
        pisa.build_pyramid_ragged(p)
        return p

    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device=DEV)
    eager, graphed = fresh_state(), fresh_state()
    ie = torch.empty(steps, B, Hkv, K, dtype=torch.int32, device=DEV)
    se = torch.empty(steps, B, Hkv, K, dtype=torch.float32, device=DEV)
    ig, sg = torch.empty_like(ie), torch.empty_like(se)
    for s in range(steps):
        pisa.decode_append_and_select(qd[s], kd[s], eager, K, workspace=ws, out=(ie[s], se[s]))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for s in range(steps):
            pisa.decode_append_and_select(qd[s], kd[s], graphed, K, workspace=ws, out=(ig[s], sg[s]))
    graph.replay()
    torch.cuda.synchronize()
    assert pisa.check_device_status(ws) == 0
    assert torch.equal(ie, ig) and torch.equal(se, sg)
    assert torch.equal(eager.lengths, graphed.lengths)
    assert torch.equal(eager.keys, graphed.keys)
    assert torch.equal(eager.summaries, graphed.summaries)
