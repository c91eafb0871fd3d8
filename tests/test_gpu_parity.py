"""CUDA path vs the fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth
import oracle

from parity import STAT_KEYS, compare_prefill, compare_decode, pyramid_tolerance, record

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _f32(x: torch.Tensor) -> np.ndarray:
    return x.float().cpu().numpy()


def _run_prefill(q, k, K, causal=True):
    qd, kd = q.to(DEV), k.to(DEV)
    pyr = pisa.build_pyramid(kd)
    B, N, Hq, _ = q.shape
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, k.shape[2], K), dtype=torch.uint8, device=DEV)
    idx, sc = pisa.select_prefill(qd, pyr, K, causal=causal, workspace=ws)
    assert pisa.check_device_status(ws) == 0, "a kernel reported a device-side error"
    return pyr, idx.cpu().numpy(), sc.cpu().numpy()


def _assert_stats(st, max_excused_frac=0.01):
    assert st["unexcused"] == 0, st["messages"]
    assert st.get("score_bad", 0) == 0, st["messages"]
    assert st["excused"] <= max_excused_frac * st["rows"] + 2, st


def test_pyramid_matches_oracle_means():
    for (B, N, Hkv, seed) in ((1, 2048, 1, 0), (2, 16421, 2, 1), (1, 200, 3, 3), (3, 64, 2, 4), (1, 1, 1, 5)):
        _, k = synth.iid(B, N, 2 * Hkv, Hkv, seed=seed)
        pyr = pisa.build_pyramid(k.to(DEV))
        torch.cuda.synchronize()
        got = pyr.summaries.double().cpu().numpy()
        want = oracle.build_pyramid(_f32(k))
        assert got.shape == want.shape
        tol = pyramid_tolerance(_f32(k))
        err = np.abs(got - want)
        assert (err <= tol).all(), f"N={N}: worst error / bound = {(err / tol).max():.3g}"


def test_tiny_all_queries():
    q, k, w = synth.make("tiny-2k")
    _, idx, sc = _run_prefill(q, k, w["K"])
    t = np.arange(w["N"])
    st = compare_prefill(idx, sc, _f32(q), _f32(k), t, w["K"])
    record("tiny-2k", st)
    _assert_stats(st)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("K", [1, 3, 16, 32])
def test_small_shapes_all_queries(causal, K):
    q, k = synth.iid(2, 1000, 8, 2, seed=7)
    _, idx, sc = _run_prefill(q, k, K, causal=causal)
    st = compare_prefill(idx, sc, _f32(q), _f32(k), np.arange(1000), K, causal=causal)
    _assert_stats(st)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_group_sizes(G):
    q, k = synth.iid(1, 3000, 2 * G, 2, seed=20 + G)
    _, idx, sc = _run_prefill(q, k, 8)
    st = compare_prefill(idx, sc, _f32(q), _f32(k), np.arange(3000), 8)
    _assert_stats(st)


@pytest.mark.parametrize("K", [2, 8])
def test_edge_lengths(K):
    # K = 8 takes the eight-lanes-per-row final Top-K, whose last block holds rows past N
    for N in (1, 2, 63, 64, 65, 127, 128, 129, 513):
        q, k = synth.iid(1, N, 4, 1, seed=N)
        _, idx, sc = _run_prefill(q, k, K)
        st = compare_prefill(idx, sc, _f32(q), _f32(k), np.arange(N), K)
        _assert_stats(st)


def test_ragged_structured_all_queries():
    q, k, w = synth.make("ragged-16421")
    _, idx, sc = _run_prefill(q, k, w["K"])
    t = np.arange(w["N"])
    st = compare_prefill(idx, sc, _f32(q), _f32(k), t, w["K"])
    record("ragged-16421", st)
    _assert_stats(st)


def test_latency_32k_all_queries():
    q, k, w = synth.make("latency-32k")
    _, idx, sc = _run_prefill(q, k, w["K"])
    t = np.arange(w["N"])
    st = compare_prefill(idx, sc, _f32(q), _f32(k), t, w["K"])
    record("latency-32k", st)
    _assert_stats(st)


def test_decode_steps_match_oracle_and_rebuild():
    B, Hq, Hkv, K, n_ctx, steps = 3, 32, 2, 8, 4030, 70  # crosses a leaf boundary and 2^6 leaves
    n_cap = n_ctx + steps
    cache, g = synth.decode_context(B, n_ctx, n_cap, Hkv, seed=2)
    cache_d = cache.to(DEV)
    pyr = pisa.Pyramid.allocate(cache_d, with_lengths=True)
    pisa.build_pyramid(pyr, N=n_ctx)
    for s in range(steps):
        qn, kn = synth.decode_step(g, B, Hq, Hkv)
        idx, sc = pisa.decode_append_and_select(qn.to(DEV), kn.to(DEV), pyr, K)
        cache[:, n_ctx + s] = kn
        if s % 7 == 0 or s == steps - 1:
            torch.cuda.synchronize()
            lengths = np.full(B, n_ctx + s + 1)
            st = compare_decode(idx.cpu().numpy(), sc.cpu().numpy(), _f32(qn), _f32(cache), lengths, K)
            _assert_stats(st)
    torch.cuda.synchronize()
    assert pyr.lengths.cpu().tolist() == [n_cap] * B
    assert torch.equal(pyr.keys.cpu(), cache)
    # the incrementally updated pyramid equals a fresh build, bit for bit
    fresh = pisa.build_pyramid(cache.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(fresh.summaries, pyr.summaries)



@pytest.mark.parametrize("G,K", [(1, 1), (2, 3), (4, 16), (8, 32), (16, 32), (16, 1), (1, 32), (4, 8)])
def test_decode_group_sizes_and_k(G, K):
    """Decode steps for every supported query-group size and K from 1 to 32 (up
    to 64 candidates per level, i.e. 16 tiles of four over the walking warps and
    the second word of the rank), each checked step compared with the oracle's
    walk of the newest query; a 12000-token context keeps levels of more than 32
    nodes."""
    B, Hkv, n_ctx, steps = 2, 2, 12000, 20
    Hq = G * Hkv
    n_cap = n_ctx + steps
    cache, g = synth.decode_context(B, n_ctx, n_cap, Hkv, seed=5 + G + K)
    pyr = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    pisa.build_pyramid(pyr, N=n_ctx)
    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device=DEV)
    for s in range(steps):
        qn, kn = synth.decode_step(g, B, Hq, Hkv)
        idx, sc = pisa.decode_append_and_select(qn.to(DEV), kn.to(DEV), pyr, K, workspace=ws)
        cache[:, n_ctx + s] = kn
        if s in (0, 9, steps - 1):
            torch.cuda.synchronize()
            assert pisa.check_device_status(ws) == 0
            lengths = np.full(B, n_ctx + s + 1)
            st = compare_decode(idx.cpu().numpy(), sc.cpu().numpy(), _f32(qn), _f32(cache), lengths, K)
            assert st["unexcused"] == 0 and st["score_bad"] == 0, st["messages"]
    torch.cuda.synchronize()
    fresh = pisa.build_pyramid(cache.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(fresh.summaries, pyr.summaries)

def test_decode_full_cache_reports_bounds():
    B, Hq, Hkv, K = 2, 8, 2, 4
    cache, g = synth.decode_context(B, 100, 100, Hkv, seed=3)
    pyr = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    pisa.build_pyramid(pyr)
    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device=DEV)
    qn, kn = synth.decode_step(g, B, Hq, Hkv)
    idx, _ = pisa.decode_append_and_select(qn.to(DEV), kn.to(DEV), pyr, K, workspace=ws)
    assert pisa.check_device_status(ws) == 6
    assert pyr.lengths.cpu().tolist() == [100, 100]
    assert (idx.cpu() == -1).all()


@pytest.mark.parametrize("name,n_sample", [("latency-64k", 65536), ("latency-128k", 65536), ("latency-256k", 65536)])
def test_latency_full_size_sampled(name, n_sample):
    """Full-size passes (the benchmark's launch configuration) checked on a seeded
    sample of query positions plus the last 1024, which the oracle walks one by one."""
    q, k, w = synth.make(name)
    _, idx, sc = _run_prefill(q, k, w["K"])
    N = w["N"]
    rng = np.random.default_rng(1234)
    n_sample = min(n_sample, N - 1024)  # 64K: every position
    t = np.unique(np.concatenate([rng.choice(N - 1024, n_sample, replace=False), np.arange(N - 1024, N)]))
    st = compare_prefill(idx[:, :, t], sc[:, :, t], _f32(q[:, t]), _f32(k), t, w["K"])
    record(name + " (sampled)", st)
    _assert_stats(st)


def test_decode_at_full_size_matches_oracle():
    """The decode workload at its own size: 16 sequences over a 131072-token
    context (2048 leaves, 12 levels); the first append makes 2049 leaves and 13
    levels, the 65th opens leaf 2049.  Each checked step is compared with the
    oracle's walk of the newest query over the keys present; at the end the
    incrementally maintained pyramid equals a fresh build bit for bit."""
    B, Hq, Hkv, K, n_ctx, steps = 16, 32, 2, 8, 131072, 70
    n_cap = n_ctx + steps
    cache, g = synth.decode_context(B, n_ctx, n_cap, Hkv, seed=2)
    pyr = pisa.Pyramid.allocate(cache.to(DEV), with_lengths=True)
    pisa.build_pyramid(pyr, N=n_ctx)
    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device=DEV)
    cache_f = _f32(cache)
    total = dict({k: 0 for k in STAT_KEYS}, score_max_rel=0.0)
    for s in range(steps):
        qn, kn = synth.decode_step(g, B, Hq, Hkv)
        idx, sc = pisa.decode_append_and_select(qn.to(DEV), kn.to(DEV), pyr, K, workspace=ws)
        cache[:, n_ctx + s] = kn
        cache_f[:, n_ctx + s] = _f32(kn)
        if s in (0, 1, 2, 31, 63, 64, 65, steps - 1):
            torch.cuda.synchronize()
            assert pisa.check_device_status(ws) == 0
            lengths = np.full(B, n_ctx + s + 1)
            st = compare_decode(idx.cpu().numpy(), sc.cpu().numpy(), _f32(qn), cache_f, lengths, K)
            _assert_stats(st, max_excused_frac=0.05)
            for k in STAT_KEYS:
                total[k] += st[k]
            total["score_max_rel"] = max(total["score_max_rel"], st["score_max_rel"])
    record("decode-16x131k", total)
    torch.cuda.synchronize()
    assert pyr.lengths.cpu().tolist() == [n_cap] * B
    fresh = pisa.build_pyramid(cache.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(fresh.summaries, pyr.summaries)
