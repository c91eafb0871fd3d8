"""Comparison of the CUDA path's selections with the fp64 oracle's.

Rules (fixed before any kernel was written):
  * index sets must match exactly, except rows where the oracle's walk met a
    near tie: at some scored level on its path the K-th best and (K+1)-th best
    scores differ by less than TIE (1e-3).  Such rows are counted and reported;
    the GPU's answer for them must still be a valid selection (ascending,
    distinct, eligible leaves, as many as the oracle selected) whose reported
    scores equal the oracle's exact scores of those same leaves;
  * scores must match within REL (2e-3) relative: |gpu - oracle| <=
    REL * max(1, |oracle|); padded slots are -inf on both sides.
"""
from __future__ import annotations

import numpy as np

import oracle

TIE = 1e-3
REL = 2e-3


def _score_ok(got, want):
    inf = np.isinf(want)
    with np.errstate(invalid="ignore"):
        close = np.abs(got - want) <= REL * np.maximum(1.0, np.abs(want))
    return np.where(inf, got == want, close)


def compare_prefill(gpu_idx, gpu_scores, q_rows, keys, t_list, K, causal=True, mode=0):
    """gpu_idx/gpu_scores: [B, Hkv, n_t, K] numpy for the positions in t_list;
    q_rows [B, n_t, Hq, d] float32; keys [B, N, Hkv, d] float32."""
    orc = oracle.select(q_rows, keys, K=K, causal=causal, t_list=t_list, mode=mode)
    return _compare(gpu_idx, gpu_scores, orc, q_rows, keys, t_list, K, causal, mode)


def compare_flat(gpu_idx, gpu_scores, q_rows, keys, t_list, K, causal=True, mode=0):
    """The flat selector against the oracle's flat selection (same rules; the
    near-tie gap is the oracle's K-th minus (K+1)-th leaf score)."""
    orc = oracle.flat_select(q_rows, keys, K=K, causal=causal, t_list=t_list, mode=mode)
    return _compare(gpu_idx, gpu_scores, orc, q_rows, keys, t_list, K, causal, mode)


def _compare(gpu_idx, gpu_scores, orc, q_rows, keys, t_list, K, causal, mode=0):
    oi, osc, gap = orc["idx"], orc["scores"], orc["min_gap"]
    same = np.all(gpu_idx == oi, axis=-1)  # [B, Hkv, n_t]
    near = gap < TIE
    bad_rows = ~same & ~near
    stats = dict(rows=int(same.size), exact=int(same.sum()), near_tie_rows=int(near.sum()),
                 excused=int((~same & near).sum()), unexcused=int(bad_rows.sum()))
    msgs = []
    if bad_rows.any():
        w = np.argwhere(bad_rows)[:5]
        for b, kv, it in w:
            msgs.append(f"mismatch b={b} kv={kv} t={t_list[it]} gpu={gpu_idx[b, kv, it].tolist()} "
                        f"oracle={oi[b, kv, it].tolist()} gap={gap[b, kv, it]:.3g}")
    # scores on exactly matching rows
    if gpu_scores is not None:
        ok = _score_ok(gpu_scores, osc) | ~same[..., None]
        stats["score_bad"] = int((~ok).sum())
        if (~ok).any():
            b, kv, it, j = np.argwhere(~ok)[0]
            msgs.append(f"score b={b} kv={kv} t={t_list[it]} slot={j} gpu={gpu_scores[b, kv, it, j]} "
                        f"oracle={osc[b, kv, it, j]}")
        fin = np.isfinite(osc)
        stats["score_max_rel"] = float(np.max(np.abs(gpu_scores[fin & same[..., None]] - osc[fin & same[..., None]])
                                              / np.maximum(1.0, np.abs(osc[fin & same[..., None]])), initial=0.0))
    # validity of the excused rows
    exc = ~same & near
    if exc.any():
        N = keys.shape[1]
        for b, kv, it in np.argwhere(exc):
            row = gpu_idx[b, kv, it]
            sel = row[row >= 0]
            t = t_list[it]
            n_el = (min(t, N - 1) // 64 + 1) if causal else -(-N // 64)
            n_want = int((oi[b, kv, it] >= 0).sum())
            valid = (len(sel) == n_want and np.all(np.diff(sel) > 0) and np.all(sel < n_el)
                     and np.all(row[len(sel):] == -1))
            if not valid:
                stats["unexcused"] += 1
                msgs.append(f"invalid excused row b={b} kv={kv} t={t} gpu={row.tolist()}")
        if gpu_scores is not None:
            lv = np.where(exc[..., None], gpu_idx, -1).astype(np.int32)
            want = oracle.leaf_scores(q_rows, keys, t_list, lv, causal=causal, mode=mode)
            ok = _score_ok(gpu_scores, want) | ~exc[..., None]
            stats["score_bad"] += int((~ok).sum())
            if (~ok).any():
                msgs.append("excused-row scores differ from the oracle's exact leaf scores")
    stats["messages"] = msgs
    return stats


def compare_decode(gpu_idx, gpu_scores, q_new, key_cache, lengths, K):
    """gpu_idx [B, Hkv, K]; lengths = tokens present (the new one included)."""
    orc = oracle.select_last(q_new, key_cache, lengths, K=K)
    B = gpu_idx.shape[0]
    # reuse the prefill comparison with n_t = 1 per sequence
    stats = dict(rows=0, exact=0, near_tie_rows=0, excused=0, unexcused=0, score_bad=0, messages=[])
    for b in range(B):
        n = int(lengths[b])
        o1 = {k: v[b:b + 1, :, None] if v.ndim >= 2 else v for k, v in orc.items()}
        o1["min_gap"] = orc["min_gap"][b:b + 1, :, None]
        s = _compare(gpu_idx[b:b + 1, :, None], None if gpu_scores is None else gpu_scores[b:b + 1, :, None],
                     o1, q_new[b:b + 1, None], key_cache[b:b + 1, :n], np.array([n - 1]), K, True)
        for k in ("rows", "exact", "near_tie_rows", "excused", "unexcused", "score_bad"):
            stats[k] += s.get(k, 0)
        stats["messages"] += s["messages"]
    return stats
