"""Comparison of the CUDA path's selections with the fp64 oracle's.

Rules (fixed before any kernel was written):
  * index sets must match exactly, except where near ties make more than one
    answer correct: wherever two candidates' scores differ by less than TIE
    (1e-3, absolute, on the head-summed score) either order is right.  A row
    whose set differs from the oracle's is accepted ("excused") only if the
    oracle's checker re-takes the walk along the GPU's leaves and finds that a
    walk breaking near ties the other way reaches exactly that set (every scored
    level keeps a near Top-K holding the set's ancestors; the leaf level keeps
    the set).  Such a row necessarily met a near tie on the oracle's own path;
    excused rows are counted and reported, and their reported scores must equal
    the oracle's exact scores of those same leaves;
  * scores must match within REL (2e-3) relative: |gpu - oracle| <=
    REL * max(1, |oracle|); padded slots are -inf on both sides.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

TIE = 1e-3
REL = 2e-3

STAT_KEYS = ("rows", "exact", "near_tie_rows", "excused", "unexcused", "undecided", "score_bad")


U32 = 2.0 ** -24  # unit roundoff of fp32


def pyramid_tolerance(keys, n=None, C=64):
    """Bound on |GPU summary - exact mean| for every node and feature.

    The GPU sums a leaf's n <= C keys in token order in fp32 and divides by n
    (error <= (n-1)u * sum|k| / n + u|mean|), then each merge of two children is
    fl(fl(fl(m0*n0) + fl(m1*n1)) / (n0+n1)): three roundings of magnitude at most
    u times the token-weighted mean of |child|, on top of the token-weighted mean
    of the children's errors.  By induction a node of level l is off by at most
    (C + 3(l-1) + 1) u times the mean of |k| over its tokens (per feature), up to
    second-order terms, which the factor 1 + 1e-3 covers.  The scale is the mean
    of |k|, not |mean|: a mean that cancels to near zero keeps the rounding
    errors of its terms, so a tolerance relative to the mean itself cannot hold.
    keys [B, n_cap, Hkv, d] float32 -> [B, Hkv, total_nodes(n), d]."""
    n = keys.shape[1] if n is None else n
    absmean = oracle.build_pyramid(np.abs(keys), n=n)
    sizes = oracle.level_sizes(n)
    lvl = np.concatenate([np.full(m, l, dtype=np.float64) for l, m in enumerate(sizes, start=1)])
    return (C + 3.0 * (lvl - 1) + 1.0)[None, None, :, None] * U32 * absmean * (1.0 + 1e-3)


def _score_ok(got, want):
    inf = np.isinf(want)
    with np.errstate(invalid="ignore"):
        close = np.abs(got - want) <= REL * np.maximum(1.0, np.abs(want))
    return np.where(inf, got == want, close)


def compare_prefill(gpu_idx, gpu_scores, q_rows, keys, t_list, K, causal=True, mode=0):
    """gpu_idx/gpu_scores: [B, Hkv, n_t, K] numpy for the positions in t_list;
    q_rows [B, n_t, Hq, d] float32; keys [B, N, Hkv, d] float32."""
    t_list = np.asarray(t_list)
    orc = oracle.select(q_rows, keys, K=K, causal=causal, t_list=t_list, mode=mode)

    def check(its):
        return oracle.check_selection(q_rows[:, its], keys, t_list[its], gpu_idx[:, :, its], K=K, tie=TIE,
                                      causal=causal, mode=mode)

    def rescore(lv):
        return oracle.leaf_scores(q_rows, keys, t_list, lv, causal=causal, mode=mode)

    return _compare(gpu_idx, gpu_scores, orc, check, rescore, t_list)


def compare_flat(gpu_idx, gpu_scores, q_rows, keys, t_list, K, causal=True, mode=0):
    """The flat selector against the oracle's flat selection (same rules; a
    differing set must be a near Top-K of all eligible leaves)."""
    t_list = np.asarray(t_list)
    orc = oracle.flat_select(q_rows, keys, K=K, causal=causal, t_list=t_list, mode=mode)

    def check(its):
        return oracle.check_selection(q_rows[:, its], keys, t_list[its], gpu_idx[:, :, its], K=K, tie=TIE,
                                      causal=causal, flat=True, mode=mode)

    def rescore(lv):
        return oracle.leaf_scores(q_rows, keys, t_list, lv, causal=causal, mode=mode)

    return _compare(gpu_idx, gpu_scores, orc, check, rescore, t_list)


def _compare(gpu_idx, gpu_scores, orc, check, rescore, t_list):
    oi, osc, gap = orc["idx"], orc["scores"], orc["min_gap"]
    same = np.all(gpu_idx == oi, axis=-1)  # [B, Hkv, n_t]
    near = gap < TIE
    verdict = np.ones(same.shape, dtype=np.int32)
    its = np.unique(np.argwhere(~same)[:, 2]) if (~same).any() else np.zeros(0, np.int64)
    if len(its):
        verdict[:, :, its] = check(its)
    exc = ~same & (verdict == 1)
    bad_rows = ~same & (verdict != 1)
    stats = dict(rows=int(same.size), exact=int(same.sum()), near_tie_rows=int(near.sum()),
                 excused=int(exc.sum()), unexcused=int(bad_rows.sum()),
                 undecided=int((~same & (verdict == -1)).sum()), score_bad=0)
    msgs = []
    for b, kv, it in np.argwhere(bad_rows)[:5]:
        msgs.append(f"mismatch b={b} kv={kv} t={t_list[it]} gpu={gpu_idx[b, kv, it].tolist()} "
                    f"oracle={oi[b, kv, it].tolist()} gap={gap[b, kv, it]:.3g} verdict={verdict[b, kv, it]}")
    # a reachable different set implies a near tie on the oracle's path
    if (exc & ~near).any():
        stats["unexcused"] += int((exc & ~near).sum())
        msgs.append("checker accepted a row whose oracle path had no near tie")
    if gpu_scores is not None:
        ok = _score_ok(gpu_scores, osc) | ~same[..., None]
        stats["score_bad"] = int((~ok).sum())
        if (~ok).any():
            b, kv, it, j = np.argwhere(~ok)[0]
            msgs.append(f"score b={b} kv={kv} t={t_list[it]} slot={j} gpu={gpu_scores[b, kv, it, j]} "
                        f"oracle={osc[b, kv, it, j]}")
        m = np.isfinite(osc) & same[..., None]
        stats["score_max_rel"] = float(np.max(np.abs(gpu_scores[m] - osc[m]) / np.maximum(1.0, np.abs(osc[m])),
                                              initial=0.0))
        if exc.any():
            lv = np.where(exc[..., None], gpu_idx, -1).astype(np.int32)
            want = rescore(lv)
            ok = _score_ok(gpu_scores, want) | ~exc[..., None]
            stats["score_bad"] += int((~ok).sum())
            if (~ok).any():
                msgs.append("excused-row scores differ from the oracle's exact leaf scores")
    stats["messages"] = msgs
    return stats


def compare_decode(gpu_idx, gpu_scores, q_new, key_cache, lengths, K):
    """gpu_idx [B, Hkv, K]; lengths = tokens present (the new one included)."""
    lengths = np.asarray(lengths)
    orc = oracle.select_last(q_new, key_cache, lengths, K=K)
    o = dict(idx=orc["idx"][:, :, None], scores=orc["scores"][:, :, None], min_gap=orc["min_gap"][:, :, None])

    def check(its):
        return oracle.check_last(q_new, key_cache, lengths, gpu_idx, K=K, tie=TIE)[:, :, None]

    def rescore(lv):
        out = np.full(lv.shape, -np.inf)
        for b in range(lv.shape[0]):
            n = int(lengths[b])
            out[b:b + 1] = oracle.leaf_scores(q_new[b:b + 1, None], key_cache[b:b + 1, :n], np.array([n - 1]),
                                              lv[b:b + 1])
        return out

    sc = None if gpu_scores is None else gpu_scores[:, :, None]
    # one row per (sequence, KV head); messages show t = -1 for "the newest query"
    return _compare(gpu_idx[:, :, None], sc, o, check, rescore, np.full(1, -1))


def record(name, stats):
    """Append one workload's counts to the JSON-lines file named by
    PISA_PARITY_LOG (when set), so that a GPU run leaves a table of rows, exact
    rows, near-tie rows and excused rows per workload."""
    path = os.environ.get("PISA_PARITY_LOG")
    line = {"workload": name, **{k: stats.get(k) for k in STAT_KEYS}}
    if "score_max_rel" in stats:
        line["score_max_rel"] = stats["score_max_rel"]
    print(name, line)
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")
