"""fp64 CPU oracle for the PISA pyramid Top-K block-selection stage.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow restatement of what
the method computes ("Block Sparse Attention with Log-Linear Complexity",
§3.1 building the pyramid, §3.2 the coarse-to-fine Top-K walk, "Scoring:
LogSumExp", §4.1 the GQA head sum).  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs may import it.  The CUDA
product path (``pyramid_top_block_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``pisa_oracle.c`` (fp64, OpenMP over queries); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Inputs are float32 arrays that hold bf16 values exactly.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pisa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def build(verbose: bool = False) -> str:
    """Compile pisa_oracle.c into a shared library (OpenMP when gcc has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, f"libpisa_oracle_{_src_hash()}.so")
    if os.path.exists(out):
        return out
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    for flags in (["-fopenmp"], []):
        cmd = base[:1] + flags + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, out)
            if verbose:
                print(" ".join(cmd))
            return out
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.pisa_oracle_num_levels.argtypes = [i64, i32, i32]
        lib.pisa_oracle_num_levels.restype = i32
        lib.pisa_oracle_level_size.argtypes = [i64, i32, i32, i32]
        lib.pisa_oracle_level_size.restype = i64
        lib.pisa_oracle_total_nodes.argtypes = [i64, i32, i32]
        lib.pisa_oracle_total_nodes.restype = i64
        lib.pisa_oracle_max_threads.argtypes = []
        lib.pisa_oracle_max_threads.restype = i32
        lib.pisa_oracle_build_pyramid.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, i32, vp]
        lib.pisa_oracle_build_pyramid.restype = i32
        lib.pisa_oracle_select.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, i32,
                                           vp, i64, vp, vp, vp, vp, i32, i32]
        lib.pisa_oracle_select.restype = i32
        lib.pisa_oracle_select_last.argtypes = [vp, vp, i32, i64, vp, i32, i32, i32, i32, i32, i32,
                                                vp, vp, vp, vp, i32]
        lib.pisa_oracle_select_last.restype = i32
        lib.pisa_oracle_leaf_scores.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, i32, i32,
                                                vp, i64, i32, vp, vp, i32, i32]
        lib.pisa_oracle_leaf_scores.restype = i32
        lib.pisa_oracle_flat_select.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, i32,
                                                vp, i64, vp, vp, vp, i32, i32]
        lib.pisa_oracle_flat_select.restype = i32
        lib.pisa_oracle_attention.argtypes = [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i64,
                                              i32, vp, vp, i32]
        lib.pisa_oracle_attention.restype = i32
        lib.pisa_oracle_node_score.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, i32, i32, i64,
                                               i32, i64, i32]
        lib.pisa_oracle_node_score.restype = dbl
        lib.pisa_oracle_check_selection.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, i32,
                                                    vp, i64, vp, dbl, i32, i32, vp, i32]
        lib.pisa_oracle_check_selection.restype = i32
        lib.pisa_oracle_check_last.argtypes = [vp, vp, i32, i64, vp, i32, i32, i32, i32, i32, i32,
                                               vp, dbl, vp, i32]
        lib.pisa_oracle_check_last.restype = i32
        _lib = lib
        return lib


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def num_levels(n: int, C: int = 64, g: int = 2) -> int:
    return int(_load().pisa_oracle_num_levels(n, C, g))


def level_sizes(n: int, C: int = 64, g: int = 2) -> list[int]:
    lib = _load()
    L = lib.pisa_oracle_num_levels(n, C, g)
    return [int(lib.pisa_oracle_level_size(n, C, g, l)) for l in range(1, L + 1)]


def total_nodes(n: int, C: int = 64, g: int = 2) -> int:
    return int(_load().pisa_oracle_total_nodes(n, C, g))


def max_threads() -> int:
    return int(_load().pisa_oracle_max_threads())


def build_pyramid(keys, n: int | None = None, C: int = 64, g: int = 2, recursive: bool = False):
    """Mean pyramid, fp64.  keys [B, n_cap, Hkv, d] -> [B, Hkv, total_nodes(n), d]."""
    k = _f32(keys)
    B, n_cap, Hkv, d = k.shape
    n = n_cap if n is None else n
    out = np.empty((B, Hkv, total_nodes(n, C, g), d), dtype=np.float64)
    rc = _load().pisa_oracle_build_pyramid(_ptr(k), B, n_cap, n, Hkv, d, C, g, int(recursive), _ptr(out))
    if rc:
        raise ValueError("oracle build_pyramid: bad arguments")
    return out


def select(q, keys, K: int, C: int = 64, g: int = 2, causal: bool = True, t_list=None,
           threads: int = 0, mode: int = 0):
    """Prefill selection.  mode: block score, 0 = LSE (PISA), 1 = mean of the
    child logits (PISA-1), 2 = mean plus half their variance (PISA-2).

    q: [B, N, Hq, d] (all positions) or [B, len(t_list), Hq, d] (rows of t_list).
    keys: [B, N, Hkv, d].  Returns dict(idx [B,Hkv,n_t,K] int32, scores fp64,
    min_gap [B,Hkv,n_t], n_scored [B,Hkv,n_t], t [n_t]).
    """
    k = _f32(keys)
    B, N, Hkv, d = k.shape
    Hq = q.shape[2]
    if t_list is None:
        t = np.arange(N, dtype=np.int64)
    else:
        t = np.ascontiguousarray(t_list, dtype=np.int64)
    qq = _f32(q)
    if qq.shape[1] != len(t):
        raise ValueError("q must hold one row per listed query position")
    n_t = len(t)
    idx = np.empty((B, Hkv, n_t, K), dtype=np.int32)
    sc = np.empty((B, Hkv, n_t, K), dtype=np.float64)
    gap = np.empty((B, Hkv, n_t), dtype=np.float64)
    ns = np.empty((B, Hkv, n_t), dtype=np.int32)
    rc = _load().pisa_oracle_select(_ptr(qq), _ptr(k), B, N, Hq, Hkv, d, C, g, K, int(causal),
                                    _ptr(t), n_t, _ptr(idx), _ptr(sc), _ptr(gap), _ptr(ns), threads, mode)
    if rc:
        raise ValueError("oracle select: bad arguments")
    return dict(idx=idx, scores=sc, min_gap=gap, n_scored=ns, t=t)


def select_last(q_new, key_cache, lengths, K: int, C: int = 64, g: int = 2, threads: int = 0):
    """Decode selection for the newest query of each sequence.

    q_new [B, Hq, d]; key_cache [B, n_cap, Hkv, d] with lengths[b] valid tokens.
    """
    k = _f32(key_cache)
    B, n_cap, Hkv, d = k.shape
    qq = _f32(q_new)
    Hq = qq.shape[1]
    ln = np.ascontiguousarray(lengths, dtype=np.int64)
    idx = np.empty((B, Hkv, K), dtype=np.int32)
    sc = np.empty((B, Hkv, K), dtype=np.float64)
    gap = np.empty((B, Hkv), dtype=np.float64)
    ns = np.empty((B, Hkv), dtype=np.int32)
    rc = _load().pisa_oracle_select_last(_ptr(qq), _ptr(k), B, n_cap, _ptr(ln), Hq, Hkv, d, C, g, K,
                                         _ptr(idx), _ptr(sc), _ptr(gap), _ptr(ns), threads)
    if rc:
        raise ValueError("oracle select_last: bad arguments")
    return dict(idx=idx, scores=sc, min_gap=gap, n_scored=ns)


def flat_select(q, keys, K: int, C: int = 64, g: int = 2, causal: bool = True, t_list=None,
                threads: int = 0, mode: int = 0):
    """Flat selection: every eligible leaf scored exactly, the K best kept
    (ties to the lower index), ascending with -1 padding.

    q: [B, n_t, Hq, d] rows of t_list (or all positions); keys: [B, N, Hkv, d].
    Returns dict(idx [B,Hkv,n_t,K] int32, scores fp64, min_gap [B,Hkv,n_t], t)."""
    k = _f32(keys)
    B, N, Hkv, d = k.shape
    Hq = q.shape[2]
    t = np.arange(N, dtype=np.int64) if t_list is None else np.ascontiguousarray(t_list, dtype=np.int64)
    qq = _f32(q)
    if qq.shape[1] != len(t):
        raise ValueError("q must hold one row per listed query position")
    n_t = len(t)
    idx = np.empty((B, Hkv, n_t, K), dtype=np.int32)
    sc = np.empty((B, Hkv, n_t, K), dtype=np.float64)
    gap = np.empty((B, Hkv, n_t), dtype=np.float64)
    rc = _load().pisa_oracle_flat_select(_ptr(qq), _ptr(k), B, N, Hq, Hkv, d, C, g, K, int(causal),
                                         _ptr(t), n_t, _ptr(idx), _ptr(sc), _ptr(gap), threads, mode)
    if rc:
        raise ValueError("oracle flat_select: bad arguments")
    return dict(idx=idx, scores=sc, min_gap=gap, t=t)


def attention(q, keys, values, idx, t_list, C: int = 64, causal: bool = True, threads: int = 0):
    """Stage-two block-sparse attention: for each listed position and query head, the
    softmax-weighted sum of the values of the keys inside the selected leaves
    idx [B, Hkv, n_t, K] (-1 skipped; keys after t masked when causal).
    q [B, n_t, Hq, d] rows of t_list; keys, values [B, N, Hkv, d].  Returns
    [B, n_t, Hq, d] float64."""
    k = _f32(keys)
    v = _f32(values)
    B, N, Hkv, d = k.shape
    qq = _f32(q)
    Hq = qq.shape[2]
    t = np.ascontiguousarray(t_list, dtype=np.int64)
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    K = ii.shape[-1]
    out = np.empty((B, len(t), Hq, d), dtype=np.float64)
    rc = _load().pisa_oracle_attention(_ptr(qq), _ptr(k), _ptr(v), B, N, Hq, Hkv, d, C, int(causal), _ptr(t),
                                       len(t), K, _ptr(ii), _ptr(out), threads)
    if rc:
        raise ValueError("oracle attention: bad arguments")
    return out


def leaf_scores(q, keys, t_list, leaves, C: int = 64, g: int = 2, causal: bool = True,
                threads: int = 0, mode: int = 0):
    """Exact head-summed raw-key LSE of given leaves for given query positions.

    q [B, n_t, Hq, d]; leaves [B, Hkv, n_t, K] int (-1 -> -inf).
    """
    k = _f32(keys)
    B, N, Hkv, d = k.shape
    qq = _f32(q)
    Hq = qq.shape[2]
    t = np.ascontiguousarray(t_list, dtype=np.int64)
    lv = np.ascontiguousarray(leaves, dtype=np.int32)
    Kc = lv.shape[-1]
    out = np.empty(lv.shape, dtype=np.float64)
    rc = _load().pisa_oracle_leaf_scores(_ptr(qq), _ptr(k), B, N, Hq, Hkv, d, C, g, int(causal),
                                         _ptr(t), len(t), Kc, _ptr(lv), _ptr(out), threads, mode)
    if rc:
        raise ValueError("oracle leaf_scores: bad arguments")
    return out


def node_score(q_row, keys, level: int, node: int, t: int, kv: int = 0, C: int = 64, g: int = 2,
               causal: bool = True, mode: int = 0) -> float:
    """Head-summed LSE score of one node for one query (q_row [Hq, d], keys [1, N, Hkv, d])."""
    k = _f32(keys)
    _, N, Hkv, d = k.shape
    qq = _f32(q_row)
    Hq = qq.shape[0]
    return float(_load().pisa_oracle_node_score(_ptr(qq), _ptr(k), N, Hq, Hkv, d, C, g, int(causal),
                                                kv, t, level, node, mode))


def check_selection(q, keys, t_list, sel, K: int, tie: float = 1e-3, C: int = 64, g: int = 2,
                    causal: bool = True, flat: bool = False, mode: int = 0, threads: int = 0):
    """Is each given leaf set one that the walk (or, with flat=True, the flat
    selector) reaches when near ties -- score differences below ``tie`` -- are
    broken either way?  The walk is re-taken along the given leaves: every
    scored level must keep a near Top-K that contains their ancestors (all
    near-Top-K completions are tried), and the leaf level must keep exactly them.

    q [B, n_t, Hq, d] rows of t_list; keys [B, N, Hkv, d]; sel [B, Hkv, n_t, K].
    Returns int32 [B, Hkv, n_t]: 1 reachable, 0 not (or malformed), -1 undecided
    (search budget exhausted)."""
    k = _f32(keys)
    B, N, Hkv, d = k.shape
    qq = _f32(q)
    Hq = qq.shape[2]
    t = np.ascontiguousarray(t_list, dtype=np.int64)
    if qq.shape[1] != len(t):
        raise ValueError("q must hold one row per listed query position")
    s = np.ascontiguousarray(sel, dtype=np.int32)
    if s.shape != (B, Hkv, len(t), K):
        raise ValueError("sel must be [B, Hkv, n_t, K]")
    out = np.empty((B, Hkv, len(t)), dtype=np.int32)
    rc = _load().pisa_oracle_check_selection(_ptr(qq), _ptr(k), B, N, Hq, Hkv, d, C, g, K, int(causal),
                                             _ptr(t), len(t), _ptr(s), float(tie), int(flat), mode,
                                             _ptr(out), threads)
    if rc:
        raise ValueError("oracle check_selection: bad arguments")
    return out


def check_last(q_new, key_cache, lengths, sel, K: int, tie: float = 1e-3, C: int = 64, g: int = 2,
               threads: int = 0):
    """``check_selection`` for decode: sequence b's newest query over its
    lengths[b] keys.  q_new [B, Hq, d]; key_cache [B, n_cap, Hkv, d];
    sel [B, Hkv, K].  Returns int32 [B, Hkv]."""
    k = _f32(key_cache)
    B, n_cap, Hkv, d = k.shape
    qq = _f32(q_new)
    Hq = qq.shape[1]
    ln = np.ascontiguousarray(lengths, dtype=np.int64)
    s = np.ascontiguousarray(sel, dtype=np.int32)
    if s.shape != (B, Hkv, K):
        raise ValueError("sel must be [B, Hkv, K]")
    out = np.empty((B, Hkv), dtype=np.int32)
    rc = _load().pisa_oracle_check_last(_ptr(qq), _ptr(k), B, n_cap, _ptr(ln), Hq, Hkv, d, C, g, K,
                                        _ptr(s), float(tie), _ptr(out), threads)
    if rc:
        raise ValueError("oracle check_last: bad arguments")
    return out
