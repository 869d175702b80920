"""Thin ctypes binding of ``libhstu.so`` (the C ABI of ``include/hstu_attn.h``).

The functions keep the C names and only marshal arguments: torch tensors or
raw integer addresses become pointers, a torch stream becomes a
``cudaStream_t``, and a negative status becomes an ``HstuError``.  Every step
of the attention runs in the library's CUDA kernel; there is no Python or
CPU fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhstu.so")

HSTU_OK = 0
HSTU_ERR_INVALID_ARG = -1
HSTU_ERR_UNSUPPORTED = -2
HSTU_ERR_CUDA = -3
HSTU_ERR_TIMEOUT = -4
HSTU_ERR_NO_MEMORY = -5
HSTU_ERR_CAPACITY = -6
HSTU_NOALLOC_MAX_ITEMS = 65536
BLOCK_M = 128
HSTU_DEBUG_UNSIGNALLED_WAIT = 1
HSTU_DEBUG_TRACE = 2
HSTU_DEBUG_NO_PAIRS = 4
HSTU_DEBUG_BWD_ROWS = 8
TRACE_EVENTS = {1: "qk_issue", 2: "pv_issue", 3: "silu_start", 4: "silu_end", 5: "epi_start",
                6: "epi_end", 7: "load_k", 8: "load_v", 9: "load_q", 10: "mma_k_ready",
                11: "mma_qk_done", 12: "mma_p_ready", 13: "mma_pv_done"}

# name -> (restype, argtypes); the exported symbols of include/hstu_attn.h
_VP, _I32P, _IP = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int)


class _Rab(ctypes.Structure):
    """struct hstu_rab"""
    _fields_ = [("timestamps", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("num_pos", ctypes.c_int),
                ("time", ctypes.c_void_p), ("num_time", ctypes.c_int)]


class _NormGate(ctypes.Structure):
    """struct hstu_norm_gate"""
    _fields_ = [("u", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("eps", ctypes.c_float)]


_RABP, _NGP = ctypes.POINTER(_Rab), ctypes.POINTER(_NormGate)
_SIGNATURES = {
    "hstu_attn_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_float, ctypes.c_float, _VP, _VP]),
    "hstu_attn_fwd_host": (ctypes.c_int, [_VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                          _VP, _VP, _VP, _VP, _VP, ctypes.c_int, _VP]),
    "hstu_attn_fwd_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                             ctypes.c_float, _VP, _VP]),
    "hstu_plan_create": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(_VP)]),
    "hstu_attn_fwd_plan": (ctypes.c_int, [_VP, _VP, _VP, _VP, ctypes.c_float, ctypes.c_float, _VP, _VP]),
    "hstu_plan_destroy": (ctypes.c_int, [_VP]),
    "hstu_plan_num_items": (ctypes.c_int, [_VP, _IP]),
    "hstu_plan_num_pairs": (ctypes.c_int, [_VP, _IP]),
    "hstu_worklist_build_pairs": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, _I32P, ctypes.c_int,
                                                 _IP]),
    "hstu_plan_worklist": (ctypes.c_int, [_VP, _I32P, ctypes.c_int, _IP]),
    "hstu_worklist_schedule": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, _I32P, _I32P,
                                              ctypes.POINTER(ctypes.c_longlong)]),
    "hstu_host_runs": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, _I32P, ctypes.c_int, _IP]),
    "hstu_worklist_build": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, _I32P, ctypes.c_int, _IP]),
    "hstu_launch_shape": (ctypes.c_int, [_VP, _IP, _IP, _IP]),
    "hstu_last_status": (ctypes.c_int, [_IP, _IP]),
    "hstu_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "hstu_set_debug_flags": (ctypes.c_int, [ctypes.c_uint32]),
    "hstu_trace_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int, _IP]),
    "hstu_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "hstu_attn_fwd_targets": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                             ctypes.c_float, _VP, _VP]),
    "hstu_plan_create_targets": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.POINTER(_VP)]),
    "hstu_plan_item_hist": (ctypes.c_int, [_VP, _I32P, ctypes.c_int, _IP]),
    "hstu_worklist_build_targets": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int, _I32P,
                                                   _I32P, ctypes.c_int, _IP]),
    "hstu_worklist_build_candidates": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int,
                                                      _I32P, _I32P, ctypes.c_int, _IP]),
    "hstu_plan_create_ex": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_uint32, ctypes.POINTER(_VP)]),
    "hstu_attn_fwd_norm_gate_plan": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_float,
                                                    ctypes.c_float, ctypes.c_float, _VP, _VP]),
    "hstu_attn_fwd_plan_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _RABP, _NGP, ctypes.c_float,
                                             ctypes.c_float, _VP, _VP]),
    "hstu_attn_fwd_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32P, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, _RABP, _NGP, ctypes.c_float,
                                        ctypes.c_float, _VP, _VP]),
    "hstu_attn_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_float, ctypes.c_float, _VP, _VP, _VP, _VP]),
    "hstu_attn_bwd_plan": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_float, ctypes.c_float, _VP,
                                          _VP, _VP, _VP]),
    "hstu_worklist_build_bwd": (ctypes.c_int, [_I32P, ctypes.c_int, ctypes.c_int, _I32P, ctypes.c_int,
                                               _IP]),
    "hstu_attn_bwd_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I32P, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, _RABP, ctypes.c_float,
                                        ctypes.c_float, _VP, _VP, _VP, _VP, _VP, _VP]),
    "hstu_worklist_build_bwd_targets": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int,
                                                       _I32P, _I32P, ctypes.c_int, _IP]),
    "hstu_attn_bwd_plan_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _RABP, ctypes.c_float,
                                             ctypes.c_float, _VP, _VP, _VP, _VP, _VP, _VP]),
    "hstu_attn_fwd_norm_gate": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_float, _VP,
                                               _I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_float, ctypes.c_float, _VP,
                                               _VP]),
}

HSTU_PLAN_NORM_GATE = 1
HSTU_PLAN_BACKWARD = 2
HSTU_PLAN_CANDIDATES_ONLY = 4
HSTU_PLAN_PAIRS = 8

_lib = None


class HstuError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {hstu_status_string(code)} (status {code})")


def lib():
    """Load libhstu.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m hstu_jagged_attention_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def exported_symbols():
    return sorted(_SIGNATURES)


def _check(code: int, where: str):
    if code != HSTU_OK:
        raise HstuError(code, where)


def _addr(x) -> int | None:
    """Device/host address of a tensor or an integer address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream or None
        return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _host_offsets(offsets) -> np.ndarray:
    if hasattr(offsets, "detach"):
        offsets = offsets.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(offsets), dtype=np.int32)


def hstu_status_string(code: int) -> str:
    return lib().hstu_status_string(int(code)).decode()


def hstu_attn_fwd(q, k, v, offsets, batch: int, heads: int, d: int, max_seqlen: int, alpha: float,
                  inv_n: float, out, stream=None) -> None:
    """Enqueue the forward on ``stream`` (default: torch's current stream).

    ``offsets`` may be a CUDA int32 tensor, a CPU tensor / numpy array (host),
    or a raw address.
    """
    keep = None
    if isinstance(offsets, int):
        off_ptr = offsets
    elif hasattr(offsets, "is_cuda") and offsets.is_cuda:
        if offsets.dtype.itemsize != 4 or not offsets.is_contiguous():
            raise ValueError("device offsets must be contiguous int32")
        off_ptr = offsets.data_ptr()
    else:
        keep = _host_offsets(offsets)
        off_ptr = keep.ctypes.data
    _check(lib().hstu_attn_fwd(_addr(q), _addr(k), _addr(v), off_ptr, int(batch), int(heads), int(d),
                               int(max_seqlen), float(alpha), float(inv_n), _addr(out),
                               _stream(stream)), "hstu_attn_fwd")


def hstu_attn_fwd_host(q, k, v, offsets, batch: int, heads: int, d: int, max_seqlen: int,
                       alpha: float, inv_n: float, out, q_dev, k_dev, v_dev, out_dev,
                       n_chunks: int = 0, stream=None) -> None:
    """The forward from host q, k, v to host out (CPU tensors, page-locked
    for overlap), staged through the caller's device tensors q_dev, k_dev,
    v_dev, out_dev, in n_chunks runs of whole sequences (0: automatic) whose
    copies overlap the kernel.  ``offsets``: host int32.  Enqueued on
    ``stream``; out is valid once the stream reaches the call's end."""
    for t in (q, k, v, out):
        if hasattr(t, "is_cuda") and t.is_cuda:
            raise ValueError("q, k, v and out must be host tensors")
    off = _host_offsets(offsets)
    _check(lib().hstu_attn_fwd_host(_addr(q), _addr(k), _addr(v), off.ctypes.data, int(batch),
                                    int(heads), int(d), int(max_seqlen), float(alpha),
                                    float(inv_n), _addr(out), _addr(q_dev), _addr(k_dev),
                                    _addr(v_dev), _addr(out_dev), int(n_chunks), _stream(stream)),
           "hstu_attn_fwd_host")


def _host_targets(num_targets, batch: int) -> np.ndarray:
    nt = _host_offsets(num_targets)
    if nt.shape != (batch,):
        raise ValueError("num_targets needs one entry per sequence")
    return nt


def hstu_attn_fwd_targets(q, k, v, offsets, num_targets, batch: int, heads: int, d: int,
                          max_seqlen: int, alpha: float, inv_n: float, out, stream=None) -> None:
    """hstu_attn_fwd with the M-FALCON candidate mask: the last num_targets[b]
    tokens of sequence b see the history and themselves only.  ``num_targets``
    is host memory (CPU tensor or numpy array), one entry per sequence."""
    keep = None
    if isinstance(offsets, int):
        off_ptr = offsets
    elif hasattr(offsets, "is_cuda") and offsets.is_cuda:
        if offsets.dtype.itemsize != 4 or not offsets.is_contiguous():
            raise ValueError("device offsets must be contiguous int32")
        off_ptr = offsets.data_ptr()
    else:
        keep = _host_offsets(offsets)
        off_ptr = keep.ctypes.data
    nt = _host_targets(num_targets, int(batch))
    _check(lib().hstu_attn_fwd_targets(_addr(q), _addr(k), _addr(v), off_ptr,
                                       nt.ctypes.data_as(_I32P), int(batch), int(heads), int(d),
                                       int(max_seqlen), float(alpha), float(inv_n), _addr(out),
                                       _stream(stream)), "hstu_attn_fwd_targets")


def _offsets_arg(offsets):
    """(address, keep-alive) for offsets given as a CUDA tensor, host data or an address."""
    if isinstance(offsets, int):
        return offsets, None
    if hasattr(offsets, "is_cuda") and offsets.is_cuda:
        if offsets.dtype.itemsize != 4 or not offsets.is_contiguous():
            raise ValueError("device offsets must be contiguous int32")
        return offsets.data_ptr(), None
    keep = _host_offsets(offsets)
    return keep.ctypes.data, keep


def _rab_struct(rab):
    """rab = (timestamps int32 device tensor, pos fp32 table, time fp32 table) or None."""
    if rab is None:
        return None
    ts, pos, time = rab
    n_pos = int(pos.numel()) if hasattr(pos, "numel") else len(pos)
    n_time = int(time.numel()) if hasattr(time, "numel") else len(time)
    return ctypes.pointer(_Rab(_addr(ts), _addr(pos), n_pos, _addr(time), n_time))


def _ng_struct(norm_gate):
    """norm_gate = (u, gamma, beta, eps) or None."""
    if norm_gate is None:
        return None
    u, gamma, beta, eps = norm_gate
    return ctypes.pointer(_NormGate(_addr(u), _addr(gamma), _addr(beta), float(eps)))


def hstu_attn_fwd_plan_ex(plan: Plan, q, k, v, alpha: float, inv_n: float, out, rab=None,
                          norm_gate=None, stream=None) -> None:
    """Every option on a plan: ``rab`` = (timestamps, pos, time), ``norm_gate`` =
    (u, gamma, beta, eps) (the plan needs HSTU_PLAN_NORM_GATE)."""
    _check(lib().hstu_attn_fwd_plan_ex(plan.handle, _addr(q), _addr(k), _addr(v), _rab_struct(rab),
                                       _ng_struct(norm_gate), float(alpha), float(inv_n), _addr(out),
                                       _stream(stream)), "hstu_attn_fwd_plan_ex")


def hstu_attn_fwd_ex(q, k, v, offsets, batch: int, heads: int, d: int, max_seqlen: int, alpha: float,
                     inv_n: float, out, num_targets=None, rab=None, norm_gate=None,
                     stream=None) -> None:
    """Every option in one call (see hstu_attn_fwd_plan_ex; num_targets host memory or None)."""
    off_ptr, keep = _offsets_arg(offsets)
    nt = None if num_targets is None else _host_targets(num_targets, int(batch))
    _check(lib().hstu_attn_fwd_ex(_addr(q), _addr(k), _addr(v), off_ptr,
                                  None if nt is None else nt.ctypes.data_as(_I32P), int(batch),
                                  int(heads), int(d), int(max_seqlen), _rab_struct(rab),
                                  _ng_struct(norm_gate), float(alpha), float(inv_n), _addr(out),
                                  _stream(stream)), "hstu_attn_fwd_ex")
    del keep


def hstu_attn_bwd(q, k, v, dout, offsets, batch: int, heads: int, d: int, max_seqlen: int,
                  alpha: float, inv_n: float, dq, dk, dv, stream=None) -> None:
    """Gradients of the forward for ``dout``: dq, dk, dv (bf16, like q) are written."""
    off_ptr, keep = _offsets_arg(offsets)
    _check(lib().hstu_attn_bwd(_addr(q), _addr(k), _addr(v), _addr(dout), off_ptr, int(batch),
                               int(heads), int(d), int(max_seqlen), float(alpha), float(inv_n),
                               _addr(dq), _addr(dk), _addr(dv), _stream(stream)), "hstu_attn_bwd")
    del keep


def hstu_attn_bwd_plan(plan: Plan, q, k, v, dout, alpha: float, inv_n: float, dq, dk, dv,
                       stream=None) -> None:
    _check(lib().hstu_attn_bwd_plan(plan.handle, _addr(q), _addr(k), _addr(v), _addr(dout),
                                    float(alpha), float(inv_n), _addr(dq), _addr(dk), _addr(dv),
                                    _stream(stream)), "hstu_attn_bwd_plan")


def hstu_attn_bwd_ex(q, k, v, dout, offsets, batch: int, heads: int, d: int, max_seqlen: int,
                     alpha: float, inv_n: float, dq, dk, dv, num_targets=None, rab=None, dpos=None,
                     dtime=None, stream=None) -> None:
    """hstu_attn_bwd with candidates (``num_targets``, host memory) and the
    bias ``rab`` = (timestamps, pos, time): dpos and dtime (fp32 device, one
    entry per table entry) receive the tables' gradients."""
    off_ptr, keep = _offsets_arg(offsets)
    nt = None if num_targets is None else _host_targets(num_targets, int(batch))
    _check(lib().hstu_attn_bwd_ex(_addr(q), _addr(k), _addr(v), _addr(dout), off_ptr,
                                  None if nt is None else nt.ctypes.data_as(_I32P), int(batch),
                                  int(heads), int(d), int(max_seqlen), _rab_struct(rab),
                                  float(alpha), float(inv_n), _addr(dq), _addr(dk), _addr(dv),
                                  _addr(dpos), _addr(dtime), _stream(stream)), "hstu_attn_bwd_ex")
    del keep


def hstu_attn_bwd_plan_ex(plan: Plan, q, k, v, dout, alpha: float, inv_n: float, dq, dk, dv,
                          rab=None, dpos=None, dtime=None, stream=None) -> None:
    _check(lib().hstu_attn_bwd_plan_ex(plan.handle, _addr(q), _addr(k), _addr(v), _addr(dout),
                                       _rab_struct(rab), float(alpha), float(inv_n), _addr(dq),
                                       _addr(dk), _addr(dv), _addr(dpos), _addr(dtime),
                                       _stream(stream)), "hstu_attn_bwd_plan_ex")


def hstu_worklist_build_bwd(host_offsets, heads: int) -> np.ndarray:
    """Host-only work list of the backward: int32 (n, 4) items (first token, length, head, kt)."""
    off = _host_offsets(host_offsets)
    batch = len(off) - 1
    n = ctypes.c_int()
    _check(lib().hstu_worklist_build_bwd(off.ctypes.data_as(_I32P), batch, int(heads), None, 0,
                                         ctypes.byref(n)), "hstu_worklist_build_bwd")
    buf = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    _check(lib().hstu_worklist_build_bwd(off.ctypes.data_as(_I32P), batch, int(heads),
                                         buf.ctypes.data_as(_I32P), n.value, ctypes.byref(n)),
           "hstu_worklist_build_bwd")
    return buf[:n.value]


def hstu_attn_fwd_norm_gate(q, k, v, u, gamma, beta, eps: float, offsets, num_targets, batch: int,
                            heads: int, d: int, max_seqlen: int, alpha: float, inv_n: float, y,
                            stream=None) -> None:
    """y = Norm(attention output) (.) u: a layer norm over each token's
    heads * d outputs with affine gamma, beta (fp32, heads * d), times u
    (bf16, like q).  ``num_targets`` is None (causal) or host memory with one
    entry per sequence (the candidate mask)."""
    off_ptr, keep = _offsets_arg(offsets)
    nt = None if num_targets is None else _host_targets(num_targets, int(batch))
    _check(lib().hstu_attn_fwd_norm_gate(_addr(q), _addr(k), _addr(v), _addr(u), _addr(gamma),
                                         _addr(beta), float(eps), off_ptr,
                                         None if nt is None else nt.ctypes.data_as(_I32P),
                                         int(batch), int(heads), int(d), int(max_seqlen),
                                         float(alpha), float(inv_n), _addr(y), _stream(stream)),
           "hstu_attn_fwd_norm_gate")
    del keep


def hstu_attn_fwd_noalloc(q, k, v, offsets, batch: int, heads: int, d: int, max_seqlen: int,
                          alpha: float, inv_n: float, out, stream=None) -> None:
    """As hstu_attn_fwd, for callers that cannot let the library allocate.

    The work list goes into a fixed device array inside the library instead
    of a per-call allocation; ``offsets`` must be host memory (a CPU tensor,
    a numpy array or a host address).  Calls in flight on the GPU at the same
    time share that array and must not overlap.
    """
    keep = None
    if isinstance(offsets, int):
        off_ptr = offsets
    else:
        if hasattr(offsets, "is_cuda") and offsets.is_cuda:
            raise ValueError("hstu_attn_fwd_noalloc takes host offsets only")
        keep = _host_offsets(offsets)
        off_ptr = keep.ctypes.data
    _check(lib().hstu_attn_fwd_noalloc(_addr(q), _addr(k), _addr(v), off_ptr, int(batch), int(heads),
                                       int(d), int(max_seqlen), float(alpha), float(inv_n),
                                       _addr(out), _stream(stream)), "hstu_attn_fwd_noalloc")


class Plan:
    """Owner of an ``hstu_plan*``; call ``hstu_plan_destroy`` or use as a context manager."""

    def __init__(self, handle: int, batch: int, heads: int, d: int, max_seqlen: int, total: int):
        self.handle = handle
        self.batch, self.heads, self.d, self.max_seqlen, self.total = batch, heads, d, max_seqlen, total

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        hstu_plan_destroy(self)

    def __del__(self):
        try:
            hstu_plan_destroy(self)
        except Exception:
            pass


def hstu_plan_create(host_offsets, batch: int, heads: int, d: int, max_seqlen: int) -> Plan:
    off = _host_offsets(host_offsets)
    if len(off) < batch + 1:
        raise ValueError("offsets needs batch + 1 entries")
    h = _VP()
    _check(lib().hstu_plan_create(off.ctypes.data_as(_I32P), int(batch), int(heads), int(d),
                                  int(max_seqlen), ctypes.byref(h)), "hstu_plan_create")
    return Plan(h.value, batch, heads, d, max_seqlen, int(off[batch]) if batch else 0)


def hstu_plan_create_targets(host_offsets, num_targets, batch: int, heads: int, d: int,
                             max_seqlen: int) -> Plan:
    """A plan with the M-FALCON candidate mask (see hstu_attn_fwd_targets)."""
    off = _host_offsets(host_offsets)
    if len(off) < batch + 1:
        raise ValueError("offsets needs batch + 1 entries")
    nt = _host_targets(num_targets, int(batch))
    h = _VP()
    _check(lib().hstu_plan_create_targets(off.ctypes.data_as(_I32P), nt.ctypes.data_as(_I32P),
                                          int(batch), int(heads), int(d), int(max_seqlen),
                                          ctypes.byref(h)), "hstu_plan_create_targets")
    return Plan(h.value, batch, heads, d, max_seqlen, int(off[batch]) if batch else 0)


def hstu_plan_create_ex(host_offsets, num_targets, batch: int, heads: int, d: int, max_seqlen: int,
                        flags: int = 0) -> Plan:
    """A plan with optional candidates (``num_targets`` None or one entry per
    sequence) and flags (HSTU_PLAN_NORM_GATE: the output stage's scratch)."""
    off = _host_offsets(host_offsets)
    if len(off) < batch + 1:
        raise ValueError("offsets needs batch + 1 entries")
    nt = None if num_targets is None else _host_targets(num_targets, int(batch))
    h = _VP()
    _check(lib().hstu_plan_create_ex(off.ctypes.data_as(_I32P),
                                     None if nt is None else nt.ctypes.data_as(_I32P), int(batch),
                                     int(heads), int(d), int(max_seqlen), int(flags),
                                     ctypes.byref(h)), "hstu_plan_create_ex")
    return Plan(h.value, batch, heads, d, max_seqlen, int(off[batch]) if batch else 0)


def hstu_attn_fwd_norm_gate_plan(plan: Plan, q, k, v, u, gamma, beta, eps: float, alpha: float,
                                 inv_n: float, y, stream=None) -> None:
    _check(lib().hstu_attn_fwd_norm_gate_plan(plan.handle, _addr(q), _addr(k), _addr(v), _addr(u),
                                              _addr(gamma), _addr(beta), float(eps), float(alpha),
                                              float(inv_n), _addr(y), _stream(stream)),
           "hstu_attn_fwd_norm_gate_plan")


def hstu_plan_item_hist(plan: Plan) -> np.ndarray:
    n = hstu_plan_num_items(plan)
    buf = np.zeros(max(n, 1), dtype=np.int32)
    got = ctypes.c_int()
    _check(lib().hstu_plan_item_hist(plan.handle, buf.ctypes.data_as(_I32P), max(n, 1),
                                     ctypes.byref(got)), "hstu_plan_item_hist")
    return buf[:got.value]


def _worklist_with_hist(name: str, host_offsets, num_targets, heads: int):
    off = _host_offsets(host_offsets)
    batch = len(off) - 1
    nt = _host_targets(num_targets, batch)
    fn = getattr(lib(), name)
    n = ctypes.c_int()
    _check(fn(off.ctypes.data_as(_I32P), nt.ctypes.data_as(_I32P), batch, int(heads), None, None, 0,
              ctypes.byref(n)), name)
    items = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    hist = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(fn(off.ctypes.data_as(_I32P), nt.ctypes.data_as(_I32P), batch, int(heads),
              items.ctypes.data_as(_I32P), hist.ctypes.data_as(_I32P), n.value, ctypes.byref(n)), name)
    return items[:n.value], hist[:n.value]


def hstu_worklist_build_targets(host_offsets, num_targets, heads: int):
    """Host-only candidate work list: (items int32 (n, 4), hist int32 (n,))."""
    return _worklist_with_hist("hstu_worklist_build_targets", host_offsets, num_targets, heads)


def hstu_worklist_build_bwd_targets(host_offsets, num_targets, heads: int):
    """Host-only work list of the backward with candidates: (items, hist)."""
    return _worklist_with_hist("hstu_worklist_build_bwd_targets", host_offsets, num_targets, heads)


def hstu_worklist_build_candidates(host_offsets, num_targets, heads: int):
    """Host-only work list of a HSTU_PLAN_CANDIDATES_ONLY plan: the candidate
    work list's items whose query block holds a candidate row."""
    return _worklist_with_hist("hstu_worklist_build_candidates", host_offsets, num_targets, heads)


def hstu_attn_fwd_plan(plan: Plan, q, k, v, alpha: float, inv_n: float, out, stream=None) -> None:
    _check(lib().hstu_attn_fwd_plan(plan.handle, _addr(q), _addr(k), _addr(v), float(alpha),
                                    float(inv_n), _addr(out), _stream(stream)), "hstu_attn_fwd_plan")


def hstu_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        h, plan.handle = plan.handle, None
        _check(lib().hstu_plan_destroy(h), "hstu_plan_destroy")


def hstu_plan_num_items(plan: Plan) -> int:
    n = ctypes.c_int()
    _check(lib().hstu_plan_num_items(plan.handle, ctypes.byref(n)), "hstu_plan_num_items")
    return n.value


def hstu_plan_num_pairs(plan: Plan) -> int:
    """Pair items of the plan (0: one CTA per work item)."""
    n = ctypes.c_int()
    _check(lib().hstu_plan_num_pairs(plan.handle, ctypes.byref(n)), "hstu_plan_num_pairs")
    return n.value


def hstu_worklist_build_pairs(host_offsets, heads: int) -> np.ndarray:
    """Host-only work list of CTA pairs (no CUDA call): int32 (n_items, 4),
    rows (first token, length, head, qp)."""
    off = _host_offsets(host_offsets)
    batch = len(off) - 1
    n = ctypes.c_int()
    _check(lib().hstu_worklist_build_pairs(off.ctypes.data_as(_I32P), batch, int(heads), None, 0,
                                           ctypes.byref(n)), "hstu_worklist_build_pairs")
    buf = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    _check(lib().hstu_worklist_build_pairs(off.ctypes.data_as(_I32P), batch, int(heads),
                                           buf.ctypes.data_as(_I32P), n.value, ctypes.byref(n)),
           "hstu_worklist_build_pairs")
    return buf[:n.value]


def hstu_worklist_schedule(cost, grid: int):
    """Host-only list schedule of a longest-first work list (no CUDA call):
    (order int32 (n,), first int32 (grid + 1,), makespan)."""
    c = np.ascontiguousarray(cost, dtype=np.int32).reshape(-1)
    order = np.zeros(max(len(c), 1), dtype=np.int32)
    first = np.zeros(max(int(grid), 0) + 1, dtype=np.int32)
    span = ctypes.c_longlong()
    _check(lib().hstu_worklist_schedule(c.ctypes.data_as(_I32P), len(c), int(grid),
                                        order.ctypes.data_as(_I32P), first.ctypes.data_as(_I32P),
                                        ctypes.byref(span)),
           "hstu_worklist_schedule")
    return order[:len(c)], first, span.value


def hstu_host_runs(offsets, n_chunks: int = 0) -> np.ndarray:
    """Host-only (no CUDA call): the runs of whole sequences
    hstu_attn_fwd_host takes, as first (int32, n_runs + 1): run c is
    sequences first[c] .. first[c + 1] - 1."""
    off = _host_offsets(offsets)
    batch = len(off) - 1
    n = ctypes.c_int()
    _check(lib().hstu_host_runs(off.ctypes.data_as(_I32P), batch, int(n_chunks), None, 0,
                                ctypes.byref(n)), "hstu_host_runs")
    first = np.zeros(n.value + 1, dtype=np.int32)
    _check(lib().hstu_host_runs(off.ctypes.data_as(_I32P), batch, int(n_chunks),
                                first.ctypes.data_as(_I32P), len(first), ctypes.byref(n)),
           "hstu_host_runs")
    return first


def hstu_plan_worklist(plan: Plan) -> np.ndarray:
    n = hstu_plan_num_items(plan)
    buf = np.zeros((max(n, 1), 4), dtype=np.int32)
    got = ctypes.c_int()
    _check(lib().hstu_plan_worklist(plan.handle, buf.ctypes.data_as(_I32P), max(n, 1),
                                    ctypes.byref(got)), "hstu_plan_worklist")
    return buf[:got.value]


def hstu_worklist_build(host_offsets, heads: int) -> np.ndarray:
    """Host-only work list (no CUDA call): int32 (n_items, 4)."""
    off = _host_offsets(host_offsets)
    batch = len(off) - 1
    n = ctypes.c_int()
    _check(lib().hstu_worklist_build(off.ctypes.data_as(_I32P), batch, int(heads), None, 0,
                                     ctypes.byref(n)), "hstu_worklist_build")
    buf = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    _check(lib().hstu_worklist_build(off.ctypes.data_as(_I32P), batch, int(heads),
                                     buf.ctypes.data_as(_I32P), n.value, ctypes.byref(n)),
           "hstu_worklist_build")
    return buf[:n.value]


def hstu_launch_shape(plan: Plan) -> tuple[int, int, int]:
    g, b, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().hstu_launch_shape(plan.handle, ctypes.byref(g), ctypes.byref(b), ctypes.byref(s)),
           "hstu_launch_shape")
    return g.value, b.value, s.value


def hstu_last_status() -> tuple[int, int]:
    """(device status, site) -- reads and clears the device status word; synchronises."""
    st, site = ctypes.c_int(), ctypes.c_int()
    _check(lib().hstu_last_status(ctypes.byref(st), ctypes.byref(site)), "hstu_last_status")
    return st.value, site.value


def hstu_set_wait_timeout_ns(ns: int) -> None:
    _check(lib().hstu_set_wait_timeout_ns(int(ns)), "hstu_set_wait_timeout_ns")


def hstu_set_debug_flags(flags: int) -> None:
    _check(lib().hstu_set_debug_flags(int(flags)), "hstu_set_debug_flags")


def hstu_trace_read(capacity: int = 32768) -> np.ndarray:
    """Pipeline trace of CTA 0 (see include/hstu_attn.h): structured array
    with fields clock, event, warp, index; read and cleared."""
    buf = np.zeros(2 * capacity, dtype=np.uint64)
    n = ctypes.c_int()
    _check(lib().hstu_trace_read(buf.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), capacity,
                                 ctypes.byref(n)), "hstu_trace_read")
    raw = buf[: 2 * n.value].reshape(-1, 2)
    out = np.zeros(n.value, dtype=[("clock", np.int64), ("event", np.int32), ("warp", np.int32),
                                   ("index", np.int64)])
    out["clock"] = raw[:, 0].astype(np.int64)
    out["event"] = (raw[:, 1] >> np.uint64(48)).astype(np.int32)
    out["warp"] = ((raw[:, 1] >> np.uint64(40)) & np.uint64(0xFF)).astype(np.int32)
    out["index"] = (raw[:, 1] & np.uint64((1 << 40) - 1)).astype(np.int64)
    return out
