"""GB300-native (sm_103a) context-parallel ring-attention forward.

A thin Python binding over the C ABI of ``libcpattn.so`` (declared in ``include/cpattn.h``):
argument marshalling only. Every step of the path (token placement, ring steps with block
skipping, online softmax, merge, write-back) runs in the library's CUDA kernels. PyTorch is
used for device memory and streams. There is no CPU fallback: if the library is not built, or
a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

CONTIGUOUS, ZIGZAG, STRIPED = 0, 1, 2
LAYOUTS = {"contiguous": CONTIGUOUS, "zigzag": ZIGZAG, "striped": STRIPED}
FULL, DIAG, SKIP = 0, 1, 2

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_lib = None

SYMBOLS = [
    "cpattn_plan", "cpattn_plan_destroy", "cpattn_workspace_size", "cpattn_ring_workspace_size", "cpattn_forward",
    "cpattn_attend", "cpattn_forward_noalloc", "cpattn_check_noalloc", "cpattn_selftest_wait_timeout_noalloc",
    "cpattn_permute", "cpattn_ring_step", "cpattn_finalize", "cpattn_merge", "cpattn_plan_counts",
    "cpattn_tile_shape", "cpattn_tile_counts", "cpattn_check", "cpattn_selftest_wait_timeout", "cpattn_last_error", "cpattn_version",
    "cpattn_backward_workspace_size", "cpattn_backward", "cpattn_forward_masked", "cpattn_backward_masked",
    "cpattn_ulysses_plan", "cpattn_ulysses_workspace_size", "cpattn_ulysses_counts", "cpattn_ulysses_forward",
    "cpattn_backward_counts", "cpattn_backward_ring_workspace_size", "cpattn_backward_begin",
    "cpattn_backward_ring_step", "cpattn_backward_finalize",
    "cpattn_allgather_workspace_size", "cpattn_allgather_counts", "cpattn_allgather_forward",
    "cpattn_allgather_gather", "cpattn_allgather_attend", "cpattn_forward_docs", "cpattn_allgather_forward_docs",
    "cpattn_dist_sizes", "cpattn_dist_begin", "cpattn_dist_step", "cpattn_dist_shift", "cpattn_dist_step_shift", "cpattn_dist_finalize",
    "cpattn_plan_set_reserved_sms",
]


class CpattnError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where} failed with status {status}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libcpattn.so (built in-tree by ``_build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libcpattn.so is not built ({_build.LIB}); run context_ring_attention_blockwise_gb300."
                           "_build.build() or __graft_entry__.build() first")
    L = ctypes.CDLL(_build.LIB)
    i, u64 = ctypes.c_int, ctypes.c_uint64
    sz = ctypes.POINTER(ctypes.c_size_t)
    L.cpattn_plan.argtypes = [_I64, i, i, i, i, i, i, ctypes.POINTER(_P)]
    L.cpattn_plan_destroy.argtypes = [_P]
    L.cpattn_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_ring_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_forward.argtypes = [_P, i, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_attend.argtypes = [_P, i, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_forward_noalloc.argtypes = [_P, i, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]
    L.cpattn_check_noalloc.argtypes = [_P]
    L.cpattn_selftest_wait_timeout_noalloc.argtypes = [u64, _P]
    L.cpattn_permute.argtypes = [_P, i, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_ring_step.argtypes = [_P, i, i, ctypes.c_float, _P, ctypes.c_size_t, _P, _P]
    L.cpattn_finalize.argtypes = [_P, i, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_merge.argtypes = [i, _I64, i, i, _P, _P, _P, _P, _P]
    L.cpattn_plan_counts.argtypes = [_P, i, _P, _P, _P, _P, _P, _P]
    L.cpattn_tile_shape.argtypes = [_P, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.cpattn_tile_counts.argtypes = [_P, i, _P, _P, _P]
    L.cpattn_check.argtypes = [_P, _P]
    L.cpattn_selftest_wait_timeout.argtypes = [_P, ctypes.c_size_t, u64, _P]
    L.cpattn_forward_masked.argtypes = [_P, i, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_backward_masked.argtypes = [_P, i, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P,
                                         ctypes.c_size_t, _P]
    L.cpattn_backward_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_backward.argtypes = [_P, i, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_backward_counts.argtypes = [_P, i, _P]
    L.cpattn_backward_ring_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_backward_begin.argtypes = [_P, i, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_backward_ring_step.argtypes = [_P, i, i, ctypes.c_float, _P, ctypes.c_size_t, _P, _P]
    L.cpattn_backward_finalize.argtypes = [_P, i, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_ulysses_plan.argtypes = [_I64, i, i, i, i, i, ctypes.POINTER(_P)]
    L.cpattn_ulysses_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_ulysses_counts.argtypes = [_P, i, _P]
    L.cpattn_ulysses_forward.argtypes = [_P, i, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_allgather_workspace_size.argtypes = [_P, i, sz]
    L.cpattn_allgather_counts.argtypes = [_P, i, _P]
    L.cpattn_allgather_forward.argtypes = [_P, i, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_allgather_gather.argtypes = [_P, i, _P, ctypes.c_size_t, _P]
    L.cpattn_forward_docs.argtypes = [_P, i, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_allgather_forward_docs.argtypes = [_P, i, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                                ctypes.c_size_t, _P]
    L.cpattn_allgather_attend.argtypes = [_P, i, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_dist_sizes.argtypes = [_P, i, i, sz, sz, sz, sz]
    L.cpattn_dist_begin.argtypes = [_P, i, i, i, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_size_t, _P]
    L.cpattn_dist_step.argtypes = [_P, i, i, i, i, ctypes.c_float, _P, ctypes.c_size_t, _P, ctypes.c_size_t, _P]
    L.cpattn_dist_shift.argtypes = [_P, i, i, _P, _P, ctypes.c_size_t, i, _P]
    L.cpattn_dist_step_shift.argtypes = [_P, i, i, i, i, ctypes.c_float, _P, _P, i, ctypes.c_size_t, _P,
                                         ctypes.c_size_t, _P]
    L.cpattn_dist_finalize.argtypes = [_P, i, i, i, _P, _P, _P, ctypes.c_size_t, _P]
    L.cpattn_plan_set_reserved_sms.argtypes = [_P, i]
    L.cpattn_last_error.restype = ctypes.c_char_p
    L.cpattn_last_error.argtypes = []
    L.cpattn_version.restype = ctypes.c_char_p
    L.cpattn_version.argtypes = []
    for name in SYMBOLS:
        if name not in ("cpattn_last_error", "cpattn_version"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status: int, where: str):
    if status != 0:
        raise CpattnError(status, where, lib().cpattn_last_error().decode())


def _layout_id(layout) -> int:
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


class Plan:
    """Host-side plan for (T, h, n_kv, d_k, n_cp, layout, causal)."""

    def __init__(self, T: int, h: int, n_kv: int, d_k: int, n_cp: int, layout, causal: bool = True):
        self.T, self.h, self.n_kv, self.d, self.n_cp = int(T), int(h), int(n_kv), int(d_k), int(n_cp)
        self.layout, self.causal = _layout_id(layout), bool(causal)
        self._h = _P()
        _check(lib().cpattn_plan(self.T, self.h, self.n_kv, self.d, self.n_cp, self.layout, int(self.causal),
                                 ctypes.byref(self._h)), "cpattn_plan")

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h is not None and self._h.value:
            lib().cpattn_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_reserved_sms(self, sms: int):
        """Leave `sms` SMs free during this plan's forward attention launches (for transfers
        running beside a ring step)."""
        _check(lib().cpattn_plan_set_reserved_sms(self._h, int(sms)), "cpattn_plan_set_reserved_sms")

    def workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_workspace_size(self._h, B, ctypes.byref(out)), "cpattn_workspace_size")
        return out.value

    def ring_workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_ring_workspace_size(self._h, B, ctypes.byref(out)), "cpattn_ring_workspace_size")
        return out.value

    def backward_workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_backward_workspace_size(self._h, B, ctypes.byref(out)), "cpattn_backward_workspace_size")
        return out.value

    def backward_ring_workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_backward_ring_workspace_size(self._h, B, ctypes.byref(out)),
               "cpattn_backward_ring_workspace_size")
        return out.value

    def allgather_workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_allgather_workspace_size(self._h, B, ctypes.byref(out)), "cpattn_allgather_workspace_size")
        return out.value

    def allgather_counts(self, B: int = 1):
        import numpy as np
        recv = np.zeros(self.n_cp, dtype=np.int64)
        _check(lib().cpattn_allgather_counts(self._h, B, recv.ctypes.data), "cpattn_allgather_counts")
        return {"bytes_recv": recv}

    def dist_sizes(self, B: int, R: int):
        """Sizes of one process's part of a multi-process ring holding R ranks: (workspace bytes,
        slot bytes, the four slot regions' offsets (K, V, positions, tiles), one rank's block bytes
        in each region)."""
        ws, slot = ctypes.c_size_t(), ctypes.c_size_t()
        off, blk = (ctypes.c_size_t * 4)(), (ctypes.c_size_t * 4)()
        _check(lib().cpattn_dist_sizes(self._h, B, R, ctypes.byref(ws), ctypes.byref(slot), off, blk),
               "cpattn_dist_sizes")
        return ws.value, slot.value, tuple(off), tuple(blk)

    def tile_shape(self):
        bq, bk = ctypes.c_int(), ctypes.c_int()
        _check(lib().cpattn_tile_shape(self._h, ctypes.byref(bq), ctypes.byref(bk)), "cpattn_tile_shape")
        return bq.value, bk.value

    def counts(self, B: int = 1):
        import numpy as np
        n = self.n_cp
        full = np.zeros((n, n), dtype=np.int64)
        diag, skip = np.zeros_like(full), np.zeros_like(full)
        pairs, kvb, half = (np.zeros(n, dtype=np.int64) for _ in range(3))
        _check(lib().cpattn_plan_counts(self._h, B, full.ctypes.data, diag.ctypes.data, skip.ctypes.data,
                                        pairs.ctypes.data, kvb.ctypes.data, half.ctypes.data), "cpattn_plan_counts")
        return {"full": full, "diag": diag, "skip": skip, "pairs": pairs, "kv_bytes_recv": kvb, "half_units": half}

    def backward_counts(self, B: int = 1):
        import numpy as np
        recv = np.zeros(self.n_cp, dtype=np.int64)
        _check(lib().cpattn_backward_counts(self._h, B, recv.ctypes.data), "cpattn_backward_counts")
        return {"bytes_recv": recv}


class UlyssesPlan(Plan):
    """Host-side plan for the head split (cpattn_ulysses_plan): n_cp virtual ranks, each with all
    T tokens of h / n_cp query heads after an all-to-all."""

    def __init__(self, T: int, h: int, n_kv: int, d_k: int, n_cp: int, causal: bool = True):
        self.T, self.h, self.n_kv, self.d, self.n_cp = int(T), int(h), int(n_kv), int(d_k), int(n_cp)
        self.layout, self.causal = CONTIGUOUS, bool(causal)
        self._h = _P()
        _check(lib().cpattn_ulysses_plan(self.T, self.h, self.n_kv, self.d, self.n_cp, int(self.causal),
                                         ctypes.byref(self._h)), "cpattn_ulysses_plan")

    def workspace_size(self, B: int) -> int:
        out = ctypes.c_size_t()
        _check(lib().cpattn_ulysses_workspace_size(self._h, B, ctypes.byref(out)), "cpattn_ulysses_workspace_size")
        return out.value

    def counts(self, B: int = 1):
        import numpy as np
        recv = np.zeros(self.n_cp, dtype=np.int64)
        _check(lib().cpattn_ulysses_counts(self._h, B, recv.ctypes.data), "cpattn_ulysses_counts")
        return {"bytes_recv": recv}


# ---- device calls (torch tensors for memory and streams) ------------------------------------

def _torch():
    import torch
    return torch


def _dev_ptr(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _P(t.data_ptr())


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return _P(s.cuda_stream)


def alloc_workspace(nbytes: int, device=None):
    """A caller-owned workspace: 1024-byte aligned bytes from the torch caching allocator."""
    torch = _torch()
    buf = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-buf.data_ptr()) % 1024
    return buf[off:off + nbytes]


def _check_inputs(plan: Plan, q, k, v):
    torch = _torch()
    B, T, h, d = q.shape
    if (T, h, d) != (plan.T, plan.h, plan.d) or tuple(k.shape) != (B, T, plan.n_kv, d) or k.shape != v.shape:
        raise ValueError("q/k/v shapes do not match the plan")
    for x, nm in ((q, "q"), (k, "k"), (v, "v")):
        if x.dtype != torch.bfloat16:
            raise ValueError(f"{nm} must be bfloat16")
    return B


def forward(q, k, v, plan: Plan, pos=None, scale: float | None = None, ws=None, out=None, lse=None, stream=None):
    """cpattn_forward: q [B,T,h,d], k/v [B,T,n_kv,d] bf16 CUDA tensors (natural order).
    Returns (o [B,T,h,d] bf16, lse [B,h,T] fp32)."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if ws is None:
        ws = alloc_workspace(plan.workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    _check(lib().cpattn_forward(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                _dev_ptr(pos, "pos"), float(scale or 0.0), _dev_ptr(out, "o"), _dev_ptr(lse, "lse"),
                                _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_forward")
    return out, lse


def ulysses_forward(q, k, v, plan: UlyssesPlan, pos=None, scale: float | None = None, ws=None, out=None, lse=None,
                    stream=None):
    """cpattn_ulysses_forward: the head split's all-to-all, per-rank attention and all-to-all
    back. Arguments and results as forward()."""
    torch = _torch()
    if not isinstance(plan, UlyssesPlan):
        raise ValueError("ulysses_forward needs a UlyssesPlan")
    B = _check_inputs(plan, q, k, v)
    if ws is None:
        ws = alloc_workspace(plan.workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    _check(lib().cpattn_ulysses_forward(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                        _dev_ptr(pos, "pos"), float(scale or 0.0), _dev_ptr(out, "o"),
                                        _dev_ptr(lse, "lse"), _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
           "cpattn_ulysses_forward")
    return out, lse


def backward(q, k, v, o, lse, dout, plan: Plan, pos=None, scale: float | None = None, ws=None, dq=None, dk=None,
             dv=None, stream=None, lo=None):
    """cpattn_backward: gradients of sum(o * dout) for the forward o, lse = forward(q, k, v, plan).
    q/o/dout [B,T,h,d], k/v [B,T,n_kv,d] bf16 and lse [B,h,T] fp32 CUDA tensors (natural order).
    lo: the per-query lower bound of forward_masked (document masks), for cpattn_backward_masked.
    Returns (dq [B,T,h,d], dk [B,T,n_kv,d], dv [B,T,n_kv,d]) bf16."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    for t, name in ((o, "o"), (dout, "dout")):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if tuple(lse.shape) != (B, plan.h, plan.T) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, h, T]")
    if ws is None:
        ws = alloc_workspace(plan.backward_workspace_size(B), q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if lo is not None:
        if tuple(lo.shape) != (plan.T,) or lo.dtype != torch.int32:
            raise ValueError("lo must be an int32 tensor of T entries")
        _check(lib().cpattn_backward_masked(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                            _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), _dev_ptr(dout, "dout"),
                                            _dev_ptr(pos, "pos"), _dev_ptr(lo, "lo"), float(scale or 0.0),
                                            _dev_ptr(dq, "dq"), _dev_ptr(dk, "dk"), _dev_ptr(dv, "dv"),
                                            _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
               "cpattn_backward_masked")
        return dq, dk, dv
    _check(lib().cpattn_backward(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(o, "o"),
                                 _dev_ptr(lse, "lse"), _dev_ptr(dout, "dout"), _dev_ptr(pos, "pos"), float(scale or 0.0),
                                 _dev_ptr(dq, "dq"), _dev_ptr(dk, "dk"), _dev_ptr(dv, "dv"), _dev_ptr(ws, "ws"),
                                 ws.numel(), _stream_ptr(stream)), "cpattn_backward")
    return dq, dk, dv


def backward_begin(q, k, v, o, lse, dout, plan: Plan, ws, pos=None, stream=None):
    """cpattn_backward_begin: placement and the backward's side data, before the ring steps."""
    B = _check_inputs(plan, q, k, v)
    _check(lib().cpattn_backward_begin(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                       _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), _dev_ptr(dout, "dout"),
                                       _dev_ptr(pos, "pos"), _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
           "cpattn_backward_begin")


def backward_ring_step(plan: Plan, B: int, step: int, ws, scale: float | None = None, compute=None, copy=None):
    _check(lib().cpattn_backward_ring_step(plan.handle, B, step, float(scale or 0.0), _dev_ptr(ws, "ws"), ws.numel(),
                                           _stream_ptr(compute), _stream_ptr(copy)), "cpattn_backward_ring_step")


def backward_finalize(plan: Plan, B: int, ws, dq, dk, dv, stream=None):
    _check(lib().cpattn_backward_finalize(plan.handle, B, _dev_ptr(dq, "dq"), _dev_ptr(dk, "dk"), _dev_ptr(dv, "dv"),
                                          _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
           "cpattn_backward_finalize")


def ring_backward(q, k, v, o, lse, dout, plan: Plan, pos=None, scale: float | None = None, ws=None, dq=None,
                  dk=None, dv=None, stream=None, copy_stream=None):
    """The backward as ring steps: begin, n_cp steps (K/V and the circulating fp32 dK/dV partial
    sums hop on a copy stream; the last hop returns each block's gradient to its owner), finalize.
    Same arguments and results as backward()."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    for t, name in ((o, "o"), (dout, "dout")):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if tuple(lse.shape) != (B, plan.h, plan.T) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, h, T]")
    if ws is None:
        ws = alloc_workspace(plan.backward_ring_workspace_size(B), q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    compute = stream if stream is not None else torch.cuda.current_stream()
    copy = copy_stream if copy_stream is not None else torch.cuda.Stream(device=q.device, priority=-1)
    backward_begin(q, k, v, o, lse, dout, plan, ws, pos=pos, stream=compute)
    for s in range(plan.n_cp):
        backward_ring_step(plan, B, s, ws, scale=scale, compute=compute, copy=copy)
    backward_finalize(plan, B, ws, dq, dk, dv, stream=compute)
    return dq, dk, dv


def forward_masked(q, k, v, plan: Plan, lo, pos=None, scale: float | None = None, ws=None, out=None, lse=None,
                   stream=None):
    """cpattn_forward_masked: like forward(), with lo [T] int32 CUDA tensor, the lowest key position
    each query may see (document masks of packed sequences: the first token of its document)."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if tuple(lo.shape) != (plan.T,) or lo.dtype != torch.int32:
        raise ValueError("lo must be an int32 tensor of T entries")
    if ws is None:
        ws = alloc_workspace(plan.workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    _check(lib().cpattn_forward_masked(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                       _dev_ptr(pos, "pos"), _dev_ptr(lo, "lo"), float(scale or 0.0),
                                       _dev_ptr(out, "o"), _dev_ptr(lse, "lse"), _dev_ptr(ws, "ws"), ws.numel(),
                                       _stream_ptr(stream)), "cpattn_forward_masked")
    return out, lse


def forward_noalloc(q, k, v, plan: Plan, pos=None, scale: float | None = None, out=None, lse=None, stream=None):
    """cpattn_forward_noalloc: the forward with the library's built-in 64 MiB device scratch, for
    callers that cannot allocate a workspace (outputs may still come from the caller). A device-side
    timeout is read afterwards by check_noalloc()."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    _check(lib().cpattn_forward_noalloc(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                        _dev_ptr(pos, "pos"), float(scale or 0.0), _dev_ptr(out, "o"),
                                        _dev_ptr(lse, "lse"), _stream_ptr(stream)), "cpattn_forward_noalloc")
    return out, lse


def check_noalloc(plan: Plan | None = None):
    """cpattn_check_noalloc: raise CpattnError if a device-side wait of the last allocation-free
    forward on the current device timed out (call after synchronising its stream)."""
    _check(lib().cpattn_check_noalloc(plan.handle if plan is not None else None), "cpattn_check_noalloc")


def selftest_wait_timeout_noalloc(timeout_ns: int, stream=None):
    _check(lib().cpattn_selftest_wait_timeout_noalloc(int(timeout_ns), _stream_ptr(stream)),
           "cpattn_selftest_wait_timeout_noalloc")


def permute(q, k, v, plan: Plan, ws, pos=None, stream=None):
    B = _check_inputs(plan, q, k, v)
    _check(lib().cpattn_permute(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                _dev_ptr(pos, "pos"), _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
           "cpattn_permute")


def attend(plan: Plan, B: int, ws, out, lse, scale: float | None = None, stream=None):
    """cpattn_attend: the attention over a workspace that ``permute`` filled."""
    _check(lib().cpattn_attend(plan.handle, B, float(scale or 0.0), _dev_ptr(out, "o"), _dev_ptr(lse, "lse"),
                               _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_attend")


def ring_step(plan: Plan, B: int, step: int, ws, scale: float | None = None, compute=None, copy=None):
    """One ring step. copy: a stream for the hop to the next step, or None: the step's own kernel
    moves the blocks (one pass uses one kind of hop throughout)."""
    _check(lib().cpattn_ring_step(plan.handle, B, step, float(scale or 0.0), _dev_ptr(ws, "ws"), ws.numel(),
                                  _stream_ptr(compute), None if copy is None else _stream_ptr(copy)),
           "cpattn_ring_step")


def finalize(plan: Plan, B: int, ws, out, lse, stream=None):
    _check(lib().cpattn_finalize(plan.handle, B, _dev_ptr(out, "o"), _dev_ptr(lse, "lse"), _dev_ptr(ws, "ws"),
                                 ws.numel(), _stream_ptr(stream)), "cpattn_finalize")


def ring_forward(q, k, v, plan: Plan, pos=None, scale: float | None = None, ws=None, out=None, lse=None,
                 stream=None, copy_stream=None):
    """The ring-faithful path: permute, n_cp ring steps, finalize. Each step's hop to the next
    runs inside the step's kernel, or on copy_stream when one is given."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if ws is None:
        ws = alloc_workspace(plan.ring_workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    compute = stream if stream is not None else torch.cuda.current_stream()
    permute(q, k, v, plan, ws, pos=pos, stream=compute)
    for s in range(plan.n_cp):
        ring_step(plan, B, s, ws, scale=scale, compute=compute, copy=copy_stream)
    finalize(plan, B, ws, out, lse, stream=compute)
    return out, lse


def allgather_forward(q, k, v, plan: Plan, pos=None, lo=None, scale: float | None = None, ws=None, out=None,
                      lse=None, stream=None):
    """cpattn_allgather_forward: the all-gather variant (every rank gathers the whole K and V, then
    one attention pass for all ranks' queries). lo: optional per-query lower bound (document masks).
    Arguments and results as forward()."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if lo is not None and (tuple(lo.shape) != (plan.T,) or lo.dtype != torch.int32):
        raise ValueError("lo must be an int32 tensor of T entries")
    if ws is None:
        ws = alloc_workspace(plan.allgather_workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    _check(lib().cpattn_allgather_forward(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                          _dev_ptr(pos, "pos"), _dev_ptr(lo, "lo"), float(scale or 0.0),
                                          _dev_ptr(out, "o"), _dev_ptr(lse, "lse"), _dev_ptr(ws, "ws"), ws.numel(),
                                          _stream_ptr(stream)), "cpattn_allgather_forward")
    return out, lse


def forward_docs(q, k, v, plan: Plan, doc, pos=None, scale: float | None = None, ws=None, out=None, lse=None,
                 stream=None, allgather: bool = False):
    """cpattn_forward_docs (or, with allgather=True, cpattn_allgather_forward_docs): the forward
    under document ids, doc [T] int32 CUDA tensor; key u is visible to query t iff doc[u] == doc[t]
    (and pos[u] <= pos[t] for a causal plan). Arguments and results as forward()."""
    torch = _torch()
    B = _check_inputs(plan, q, k, v)
    if tuple(doc.shape) != (plan.T,) or doc.dtype != torch.int32:
        raise ValueError("doc must be an int32 tensor of T entries")
    if ws is None:
        ws = alloc_workspace(plan.allgather_workspace_size(B) if allgather else plan.workspace_size(B), q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, plan.h, plan.T), dtype=torch.float32, device=q.device)
    fn = lib().cpattn_allgather_forward_docs if allgather else lib().cpattn_forward_docs
    _check(fn(plan.handle, B, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(pos, "pos"),
              _dev_ptr(doc, "doc"), float(scale or 0.0), _dev_ptr(out, "o"), _dev_ptr(lse, "lse"), _dev_ptr(ws, "ws"),
              ws.numel(), _stream_ptr(stream)),
           "cpattn_allgather_forward_docs" if allgather else "cpattn_forward_docs")
    return out, lse


def allgather_gather(plan: Plan, B: int, ws, stream=None):
    _check(lib().cpattn_allgather_gather(plan.handle, B, _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)),
           "cpattn_allgather_gather")


def allgather_attend(plan: Plan, B: int, ws, out, lse, scale: float | None = None, stream=None):
    _check(lib().cpattn_allgather_attend(plan.handle, B, float(scale or 0.0), _dev_ptr(out, "o"), _dev_ptr(lse, "lse"),
                                         _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_allgather_attend")


def dist_begin(plan: Plan, B: int, rank0: int, R: int, q, k, v, ws, slot, pos=None, stream=None, lo=None):
    """cpattn_dist_begin: this process's R ranks' tokens (rank-major, each rank's local order);
    lo: their per-query lower bounds (document masks) or None."""
    _check(lib().cpattn_dist_begin(plan.handle, B, rank0, R, _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                   _dev_ptr(pos, "pos"), _dev_ptr(lo, "lo"), _dev_ptr(ws, "ws"), ws.numel(),
                                   _dev_ptr(slot, "slot"), slot.numel(), _stream_ptr(stream)), "cpattn_dist_begin")


def dist_step(plan: Plan, B: int, rank0: int, R: int, step: int, slot, ws, scale: float | None = None, stream=None):
    _check(lib().cpattn_dist_step(plan.handle, B, rank0, R, step, float(scale or 0.0), _dev_ptr(slot, "slot"),
                                  slot.numel(), _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_dist_step")


def dist_step_shift(plan: Plan, B: int, rank0: int, R: int, step: int, slot, next_slot, wrap: bool, ws,
                    scale: float | None = None, stream=None):
    """cpattn_dist_step_shift: the step on slot, and the shift from slot into next_slot done by the
    step's kernel (K, V) and copies after it (position tables), all on one stream."""
    _check(lib().cpattn_dist_step_shift(plan.handle, B, rank0, R, step, float(scale or 0.0), _dev_ptr(slot, "slot"),
                                        _dev_ptr(next_slot, "next_slot"), int(bool(wrap)), slot.numel(),
                                        _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_dist_step_shift")


def dist_shift(plan: Plan, B: int, R: int, src_slot, dst_slot, wrap: bool, stream=None):
    _check(lib().cpattn_dist_shift(plan.handle, B, R, _dev_ptr(src_slot, "src_slot"), _dev_ptr(dst_slot, "dst_slot"),
                                   dst_slot.numel(), int(bool(wrap)), _stream_ptr(stream)), "cpattn_dist_shift")


def dist_finalize(plan: Plan, B: int, rank0: int, R: int, ws, out, lse, stream=None):
    _check(lib().cpattn_dist_finalize(plan.handle, B, rank0, R, _dev_ptr(out, "o"), _dev_ptr(lse, "lse"),
                                      _dev_ptr(ws, "ws"), ws.numel(), _stream_ptr(stream)), "cpattn_dist_finalize")


def merge(o_parts, lse_parts, out=None, lse=None, stream=None):
    """cpattn_merge: o_parts [S,rows,h,d] fp32, lse_parts [S,h,rows] fp32 -> (o bf16 [rows,h,d], lse [h,rows])."""
    torch = _torch()
    S, rows, h, d = o_parts.shape
    if out is None:
        out = torch.empty((rows, h, d), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((h, rows), dtype=torch.float32, device=o_parts.device)
    _check(lib().cpattn_merge(S, rows, h, d, _dev_ptr(o_parts, "o_parts"), _dev_ptr(lse_parts, "lse_parts"),
                              _dev_ptr(out, "o"), _dev_ptr(lse, "lse"), _stream_ptr(stream)), "cpattn_merge")
    return out, lse


def tile_counts(plan: Plan, B: int, ws):
    """Tiles the kernels computed (all batch elements and heads), by (rank, step): (full, diag)."""
    import numpy as np
    full = np.zeros((plan.n_cp, plan.n_cp), dtype=np.int64)
    diag = np.zeros_like(full)
    _check(lib().cpattn_tile_counts(plan.handle, B, _dev_ptr(ws, "ws"), full.ctypes.data, diag.ctypes.data),
           "cpattn_tile_counts")
    return full, diag


def check(plan: Plan | None, ws):
    """Raise CpattnError if a device-side wait of the kernels that used ``ws`` timed out."""
    _check(lib().cpattn_check(plan.handle if plan is not None else None, _dev_ptr(ws, "ws")), "cpattn_check")


def selftest_wait_timeout(ws, timeout_ns: int, stream=None):
    _check(lib().cpattn_selftest_wait_timeout(_dev_ptr(ws, "ws"), ws.numel(), int(timeout_ns), _stream_ptr(stream)),
           "cpattn_selftest_wait_timeout")


def version() -> str:
    return lib().cpattn_version().decode()
