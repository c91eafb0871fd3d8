"""GB300-native PISA pyramid Top-K block selection.

Thin Python binding over the C ABI of ``include/pisa.h`` (library
``_build/libpisa.so``, built in-tree by ``build.py``).  This module only
marshals arguments: PyTorch provides device memory and the current CUDA
stream; every step of the selection runs in the library's CUDA kernels.  There
is no CPU fallback: if the library cannot be loaded, every call raises.

Method: "Block Sparse Attention with Log-Linear Complexity" (§3.1 pyramid of
mean-pooled keys, §3.2 coarse-to-fine Top-K walk, "Scoring: LogSumExp", §4.1
GQA head sum, §5.1 prefill and decoding kernels).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

__all__ = [
    "PisaError", "Pyramid", "load", "num_levels", "pyramid_nodes", "level_offset",
    "build_pyramid", "select_workspace_bytes", "select_prefill", "select_prefill_noalloc",
    "noalloc_prepare", "noalloc_device_status",
    "decode_workspace_bytes",
    "decode_append_and_select", "check_device_status", "status_string", "kernel_launches",
    "prefill_phases", "set_phase_events", "D", "C", "G_MERGE",
]

D, C, G_MERGE = 64, 64, 2

_lib = None


class PisaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load(path: str | None = None):
    """Load (building first if needed) the CUDA library and declare its ABI."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.LIB if os.path.exists(_build.LIB) else _build.build()
    lib = ctypes.CDLL(path)
    i32, i64, sz, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    lib.pisa_num_levels.argtypes = [i64, i32, i32]
    lib.pisa_num_levels.restype = i32
    lib.pisa_pyramid_nodes.argtypes = [i64, i32, i32]
    lib.pisa_pyramid_nodes.restype = i64
    lib.pisa_level_offset.argtypes = [i64, i32, i32, i32]
    lib.pisa_level_offset.restype = i64
    lib.pisa_build_pyramid.argtypes = [vp, i64, vp]
    lib.pisa_build_pyramid.restype = i32
    lib.pisa_select_workspace_bytes.argtypes = [i32, i64, i32, i32, i32]
    lib.pisa_select_workspace_bytes.restype = sz
    lib.pisa_select_prefill.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, vp, sz, vp]
    lib.pisa_select_prefill.restype = i32
    lib.pisa_flat_workspace_bytes.argtypes = [i32, i64, i32, i32, i32]
    lib.pisa_flat_workspace_bytes.restype = sz
    lib.pisa_select_flat.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, vp, sz, vp]
    lib.pisa_select_flat.restype = i32
    lib.pisa_select_prefill_ex.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, vp, sz, vp, i32]
    lib.pisa_select_prefill_ex.restype = i32
    lib.pisa_select_prefill_host.argtypes = [vp, vp, i64, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp, vp]
    lib.pisa_select_prefill_host.restype = i32
    lib.pisa_selftest_bounded_wait.argtypes = [vp, sz, i64, vp]
    lib.pisa_selftest_bounded_wait.restype = i32
    lib.pisa_select_flat_ex.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, vp, sz, vp, i32]
    lib.pisa_select_flat_ex.restype = i32
    lib.pisa_sparse_attention.argtypes = [vp, i32, vp, vp, i32, i64, i32, vp, i32, i32, vp, vp]
    lib.pisa_sparse_attention.restype = i32
    lib.pisa_build_pyramid_ragged.argtypes = [vp, vp]
    lib.pisa_build_pyramid_ragged.restype = i32
    lib.pisa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.pisa_decode_workspace_bytes.restype = sz
    lib.pisa_decode_append_and_select.argtypes = [vp, vp, i32, vp, i32, vp, vp, vp, sz, vp]
    lib.pisa_decode_append_and_select.restype = i32
    lib.pisa_check_device_status.argtypes = [vp, vp]
    lib.pisa_check_device_status.restype = i32
    lib.pisa_status_string.argtypes = [i32]
    lib.pisa_status_string.restype = ctypes.c_char_p
    lib.pisa_kernel_launches.argtypes = []
    lib.pisa_kernel_launches.restype = ctypes.c_uint64
    lib.pisa_set_phase_events.argtypes = [ctypes.c_void_p, i32]
    lib.pisa_set_phase_events.restype = i32
    lib.pisa_prefill_phase_count.argtypes = []
    lib.pisa_prefill_phase_count.restype = i32
    lib.pisa_prefill_phase_name.argtypes = [i32]
    lib.pisa_prefill_phase_name.restype = ctypes.c_char_p
    lib.pisa_select_prefill_noalloc.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, vp]
    lib.pisa_select_prefill_noalloc.restype = i32
    lib.pisa_noalloc_prepare.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    lib.pisa_noalloc_prepare.restype = i32
    lib.pisa_noalloc_device_status.argtypes = [vp]
    lib.pisa_noalloc_device_status.restype = i32
    lib.pisa_event_elapsed_ms.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_float)]
    lib.pisa_event_elapsed_ms.restype = i32
    _lib = lib
    return lib


class _PyrStruct(ctypes.Structure):
    _fields_ = [
        ("summaries", ctypes.c_void_p),
        ("keys", ctypes.c_void_p),
        ("lengths", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int),
        ("C", ctypes.c_int),
        ("g", ctypes.c_int),
        ("n_cap", ctypes.c_int),
    ]


def status_string(status: int) -> str:
    return load().pisa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise PisaError(status, what)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def num_levels(n: int) -> int:
    return int(load().pisa_num_levels(n, C, G_MERGE))


def pyramid_nodes(n_cap: int) -> int:
    return int(load().pisa_pyramid_nodes(n_cap, C, G_MERGE))


def level_offset(n_cap: int, level: int) -> int:
    return int(load().pisa_level_offset(n_cap, C, G_MERGE, level))


@dataclass
class Pyramid:
    """Caller-owned pyramid storage: borrowed keys [B, n_cap, Hkv, 64] bf16,
    summaries [B, Hkv, nodes(n_cap), 64] fp32 and optional lengths [B] int32."""

    keys: torch.Tensor
    summaries: torch.Tensor
    lengths: torch.Tensor | None = None

    @classmethod
    def allocate(cls, keys: torch.Tensor, with_lengths: bool = False) -> "Pyramid":
        if keys.dtype != torch.bfloat16 or keys.dim() != 4 or not keys.is_cuda:
            raise ValueError("keys must be a CUDA bf16 tensor [B, n_cap, Hkv, d]")
        B, n_cap, Hkv, d = keys.shape
        nodes = pyramid_nodes(n_cap)
        summ = torch.empty(B, Hkv, nodes, d, dtype=torch.float32, device=keys.device)
        lengths = torch.zeros(B, dtype=torch.int32, device=keys.device) if with_lengths else None
        return cls(keys.contiguous(), summ, lengths)

    @property
    def B(self):
        return self.keys.shape[0]

    @property
    def n_cap(self):
        return self.keys.shape[1]

    @property
    def Hkv(self):
        return self.keys.shape[2]

    def struct(self) -> _PyrStruct:
        return _PyrStruct(self.summaries.data_ptr(), self.keys.data_ptr(),
                          self.lengths.data_ptr() if self.lengths is not None else None,
                          self.B, self.Hkv, self.keys.shape[3], C, G_MERGE, self.n_cap)

    def level(self, level: int, n: int | None = None) -> torch.Tensor:
        """View of the summaries of one level [B, Hkv, M_level(n), d]."""
        n = self.n_cap if n is None else n
        off = level_offset(self.n_cap, level)
        m = -(-n // (C << (level - 1)))
        return self.summaries[:, :, off:off + m]


def build_pyramid(keys: torch.Tensor | Pyramid, N: int | None = None, with_lengths: bool = False,
                  stream=None) -> Pyramid:
    """Mean pyramid over the first N tokens (§3.1).  Accepts raw keys or a Pyramid."""
    pyr = keys if isinstance(keys, Pyramid) else Pyramid.allocate(keys, with_lengths)
    N = pyr.n_cap if N is None else N
    st = pyr.struct()
    _check(load().pisa_build_pyramid(ctypes.byref(st), N, _stream(stream)), "pisa_build_pyramid")
    return pyr


def select_workspace_bytes(B: int, N: int, Hq: int, Hkv: int, K: int) -> int:
    return int(load().pisa_select_workspace_bytes(B, N, Hq, Hkv, K))


def select_prefill(Q: torch.Tensor, pyr: Pyramid, K: int, causal: bool = True, N: int | None = None,
                   with_scores: bool = True, workspace: torch.Tensor | None = None,
                   out: tuple | None = None, stream=None, mode: int = 0):
    """Coarse-to-fine Top-K for every query (§3.2).  mode: block score, 0 = LSE,
    1 = mean of the child logits (PISA-1), 2 = mean + half their variance (PISA-2).

    Q [B, N, Hq, 64] bf16 (CUDA).  Returns (idx [B, Hkv, N, K] int32, scores
    [B, Hkv, N, K] fp32 or None).
    """
    if Q.dtype != torch.bfloat16 or not Q.is_cuda or Q.dim() != 4:
        raise ValueError("Q must be a CUDA bf16 tensor [B, N, Hq, d]")
    B, NQ, Hq, _ = Q.shape
    N = NQ if N is None else N
    lib = load()
    need = lib.pisa_select_workspace_bytes(B, N, Hq, pyr.Hkv, K)
    if need == 0:
        _check(2, "pisa_select_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    if out is None:
        idx = torch.empty(B, pyr.Hkv, N, K, dtype=torch.int32, device=Q.device)
        scores = torch.empty(B, pyr.Hkv, N, K, dtype=torch.float32, device=Q.device) if with_scores else None
    else:
        idx, scores = out
    st = pyr.struct()
    _check(lib.pisa_select_prefill_ex(_ptr(Q), Hq, ctypes.byref(st), N, K, int(causal), _ptr(idx),
                                      _ptr(scores), _ptr(workspace), workspace.numel(), _stream(stream),
                                      int(mode)),
           "pisa_select_prefill_ex")
    return idx, scores


_COPY_STREAMS: dict = {}


def select_prefill_host(q_host: torch.Tensor, k_host: torch.Tensor, pyr: Pyramid, K: int, causal: bool = True,
                        idx_host: torch.Tensor | None = None, q_dev: torch.Tensor | None = None,
                        idx_dev: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None, copy_stream=None) -> torch.Tensor:
    """Pyramid build + prefill selection for host-resident Q [B, N, Hq, 64] and K
    [B, N, Hkv, 64] (bf16, pinned for overlap): the library copies K into pyr.keys and
    Q into q_dev in runs of query chunks on copy_stream while `stream` selects, and
    copies each run's indices back into idx_host [B, Hkv, N, K] (int32, pinned) as soon
    as they are final.  Asynchronous: synchronise `stream` before reading idx_host.
    The device staging buffers are allocated here when not given.
    """
    if q_host.dtype != torch.bfloat16 or k_host.dtype != torch.bfloat16 or q_host.is_cuda or k_host.is_cuda:
        raise ValueError("q_host and k_host must be host bf16 tensors")
    if q_host.dim() != 4 or k_host.dim() != 4 or not q_host.is_contiguous() or not k_host.is_contiguous():
        raise ValueError("q_host [B, N, Hq, d] and k_host [B, N, Hkv, d] must be contiguous")
    B, N, Hq, _ = q_host.shape
    if k_host.shape[0] != B or k_host.shape[1] != N or k_host.shape[2] != pyr.Hkv:
        raise ValueError("k_host must be [B, N, Hkv, d] with the pyramid's B and Hkv")
    dev = pyr.keys.device
    lib = load()
    need = lib.pisa_select_workspace_bytes(B, N, Hq, pyr.Hkv, K)
    if need == 0:
        _check(2, "pisa_select_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if q_dev is None:
        q_dev = torch.empty(B, N, Hq, q_host.shape[3], dtype=torch.bfloat16, device=dev)
    if idx_dev is None:
        idx_dev = torch.empty(B, pyr.Hkv, N, K, dtype=torch.int32, device=dev)
    if idx_host is None:
        idx_host = torch.empty(B, pyr.Hkv, N, K, dtype=torch.int32, pin_memory=True)
    if copy_stream is None:  # a side stream of the library's own, one per device
        copy_stream = _COPY_STREAMS.get(dev.index)
        if copy_stream is None:
            copy_stream = _COPY_STREAMS[dev.index] = torch.cuda.Stream(device=dev)
    st = pyr.struct()
    _check(lib.pisa_select_prefill_host(ctypes.byref(st), _ptr(k_host), N, _ptr(q_host), _ptr(q_dev), Hq, K,
                                        int(causal), _ptr(idx_host), _ptr(idx_dev), _ptr(workspace),
                                        workspace.numel(), _stream(stream), _stream(copy_stream)),
           "pisa_select_prefill_host")
    return idx_host


def flat_workspace_bytes(B: int, N: int, Hq: int, Hkv: int, K: int) -> int:
    return int(load().pisa_flat_workspace_bytes(B, N, Hq, Hkv, K))


def build_pyramid_ragged(pyr: Pyramid, stream=None) -> Pyramid:
    """Build every sequence over its own length pyr.lengths[b] (set by the caller)."""
    if pyr.lengths is None:
        raise ValueError("a ragged build needs a Pyramid with lengths")
    st = pyr.struct()
    _check(load().pisa_build_pyramid_ragged(ctypes.byref(st), _stream(stream)), "pisa_build_pyramid_ragged")
    return pyr


def select_flat(Q: torch.Tensor, pyr: Pyramid, K: int, causal: bool = True, N: int | None = None,
                with_scores: bool = True, workspace: torch.Tensor | None = None,
                out: tuple | None = None, stream=None, mode: int = 0):
    """Flat selection: every eligible leaf scored exactly, the K best kept.
    Same arguments and outputs as select_prefill (only pyr.keys is read)."""
    if Q.dtype != torch.bfloat16 or not Q.is_cuda or Q.dim() != 4:
        raise ValueError("Q must be a CUDA bf16 tensor [B, N, Hq, d]")
    B, NQ, Hq, _ = Q.shape
    N = NQ if N is None else N
    lib = load()
    if workspace is None:
        need = lib.pisa_flat_workspace_bytes(B, N, Hq, pyr.Hkv, K)
        if need == 0:
            _check(2, "pisa_flat_workspace_bytes")
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    if out is None:
        idx = torch.empty(B, pyr.Hkv, N, K, dtype=torch.int32, device=Q.device)
        scores = torch.empty(B, pyr.Hkv, N, K, dtype=torch.float32, device=Q.device) if with_scores else None
    else:
        idx, scores = out
    st = pyr.struct()
    _check(lib.pisa_select_flat_ex(_ptr(Q), Hq, ctypes.byref(st), N, K, int(causal), _ptr(idx),
                                   _ptr(scores), _ptr(workspace), workspace.numel(), _stream(stream),
                                   int(mode)),
           "pisa_select_flat_ex")
    return idx, scores


def sparse_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, idx: torch.Tensor, causal: bool = True,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Stage-two block-sparse attention over the blocks in idx [B, Hkv, N, Ksel].
    Q [B, N, Hq, 64], K and V [B, N, Hkv, 64] bf16 CUDA; returns fp32 [B, N, Hq, 64]."""
    for x in (Q, K, V):
        if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 4 or not x.is_contiguous():
            raise ValueError("Q, K, V must be contiguous CUDA bf16 tensors [B, N, H, d]")
    if idx.dtype != torch.int32 or not idx.is_contiguous():
        raise ValueError("idx must be contiguous int32 [B, Hkv, N, Ksel]")
    B, N, Hq, d = Q.shape
    if out is None:
        out = torch.empty(B, N, Hq, d, dtype=torch.float32, device=Q.device)
    _check(load().pisa_sparse_attention(_ptr(Q), Hq, _ptr(K), _ptr(V), B, N, K.shape[2], _ptr(idx), idx.shape[-1],
                                        int(causal), _ptr(out), _stream(stream)),
           "pisa_sparse_attention")
    return out


def select_prefill_noalloc(Q: torch.Tensor, pyr: Pyramid, K: int, causal: bool = True,
                           with_scores: bool = True, out: tuple | None = None, stream=None):
    """select_prefill without a workspace: the library's built-in 32 MiB device
    scratch is used instead (for callers that cannot allocate device memory).
    Calls sharing that scratch must not overlap on the GPU."""
    B, N, Hq, _ = Q.shape
    if out is None:
        idx = torch.empty(B, pyr.Hkv, N, K, dtype=torch.int32, device=Q.device)
        scores = torch.empty(B, pyr.Hkv, N, K, dtype=torch.float32, device=Q.device) if with_scores else None
    else:
        idx, scores = out
    st = pyr.struct()
    _check(load().pisa_select_prefill_noalloc(_ptr(Q), Hq, ctypes.byref(st), N, K, int(causal), _ptr(idx),
                                              _ptr(scores), _stream(stream)),
           "pisa_select_prefill_noalloc")
    return idx, scores


def noalloc_prepare() -> int:
    """Set-up for select_prefill_noalloc on the current device (loads the library's
    device code there, which is when its scratch array comes into being); returns
    the scratch's device address."""
    p = ctypes.c_void_p()
    _check(load().pisa_noalloc_prepare(ctypes.byref(p)), "pisa_noalloc_prepare")
    return int(p.value or 0)


def noalloc_device_status(stream=None) -> int:
    """Synchronise the stream and return the status word of the last
    select_prefill_noalloc call on the current device (0 = ok)."""
    return int(load().pisa_noalloc_device_status(_stream(stream)))


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, K: int) -> int:
    return int(load().pisa_decode_workspace_bytes(B, Hq, Hkv, K))


def decode_append_and_select(q_new: torch.Tensor, k_new: torch.Tensor, pyr: Pyramid, K: int,
                             with_scores: bool = True, workspace: torch.Tensor | None = None,
                             out: tuple | None = None, stream=None):
    """One decoding step: append k_new at lengths[b], refresh that leaf and its
    ancestors, then select for q_new.  Returns (idx [B, Hkv, K], scores)."""
    if pyr.lengths is None:
        raise ValueError("decode needs a Pyramid with lengths")
    B, Hq, _ = q_new.shape
    lib = load()
    need = lib.pisa_decode_workspace_bytes(B, Hq, pyr.Hkv, K)
    if need == 0:
        _check(2, "pisa_decode_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_new.device)
    if out is None:
        idx = torch.empty(B, pyr.Hkv, K, dtype=torch.int32, device=q_new.device)
        scores = torch.empty(B, pyr.Hkv, K, dtype=torch.float32, device=q_new.device) if with_scores else None
    else:
        idx, scores = out
    st = pyr.struct()
    _check(lib.pisa_decode_append_and_select(_ptr(q_new), _ptr(k_new), Hq, ctypes.byref(st), K, _ptr(idx),
                                             _ptr(scores), _ptr(workspace), workspace.numel(),
                                             _stream(stream)),
           "pisa_decode_append_and_select")
    return idx, scores


def kernel_launches() -> int:
    """Kernels the library has launched since it was loaded."""
    return int(load().pisa_kernel_launches())


def prefill_phases() -> list[str]:
    lib = load()
    return [lib.pisa_prefill_phase_name(i).decode() for i in range(lib.pisa_prefill_phase_count())]


def set_phase_events(events: list | None) -> None:
    """Attach torch.cuda.Event objects recorded at the prefill phase boundaries
    (len = number of phases + 1), or None to detach."""
    lib = load()
    if not events:
        _check(lib.pisa_set_phase_events(None, 0), "pisa_set_phase_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    set_phase_events._keep = arr
    _check(lib.pisa_set_phase_events(arr, len(events)), "pisa_set_phase_events")


def event_elapsed_ms(start, end) -> float:
    """Milliseconds between two torch.cuda.Event objects, either of which may
    have been recorded by the library (phase events)."""
    out = ctypes.c_float()
    _check(load().pisa_event_elapsed_ms(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(end.cuda_event),
                                        ctypes.byref(out)), "pisa_event_elapsed_ms")
    return float(out.value)


def selftest_bounded_wait(workspace: torch.Tensor, delay_cycles: int = 2_000_000, stream=None) -> None:
    """Make a kernel's bounded barrier wait run out (nothing arrives; an abort flag goes
    up after delay_cycles): its status word in `workspace` then reads the timeout code."""
    _check(load().pisa_selftest_bounded_wait(_ptr(workspace), workspace.numel(), int(delay_cycles), _stream(stream)),
           "pisa_selftest_bounded_wait")


def check_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the kernels' status word (0 = ok)."""
    return int(load().pisa_check_device_status(_ptr(workspace), _stream(stream)))
