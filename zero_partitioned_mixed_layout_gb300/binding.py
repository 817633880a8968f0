"""Thin Python binding of libzero_pml.so (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of the optimizer step: PyTorch tensors are reduced to device
pointers and element counts, and every step of the path runs in the CUDA
kernels of the library.  There is no fallback: if the library is missing or
was not built for this GPU, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero_pml.so")

ZERO_OK = 0
ZERO_ECAPTURE = -9
ZERO_F16, ZERO_BF16, ZERO_F32 = 0, 1, 2
STATE_BYTES = 64


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {zero_strerror(code)} (code {code})")


class _Frag(ctypes.Structure):
    _fields_ = [("tensor", ctypes.c_int64), ("tensor_offset", ctypes.c_int64),
                ("rank", ctypes.c_int64), ("shard_offset", ctypes.c_int64),
                ("length", ctypes.c_int64)]


class _State(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("found_inf", ctypes.c_double),
                ("loss_scale", ctypes.c_double), ("step", ctypes.c_int64),
                ("good_steps", ctypes.c_int64), ("skipped", ctypes.c_int64),
                ("last_norm", ctypes.c_double), ("last_clip", ctypes.c_float),
                ("last_skipped", ctypes.c_int32)]


class _HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("max_norm", ctypes.c_double),
                ("min_scale", ctypes.c_double), ("scale_window", ctypes.c_int64)]


class _TList(ctypes.Structure):
    _fields_ = [("ptrs", ctypes.POINTER(ctypes.c_void_p)),
                ("numel", ctypes.POINTER(ctypes.c_int64)),
                ("n", ctypes.c_int64), ("dtype", ctypes.c_int32)]


assert ctypes.sizeof(_State) == STATE_BYTES

_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        so = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        so.zero_strerror.argtypes = [ctypes.c_int]
        so.zero_strerror.restype = ctypes.c_char_p
        so.zero_partition_layout.argtypes = [ctypes.POINTER(i64), i64, i32, i64,
                                             ctypes.POINTER(i64), ctypes.POINTER(i64),
                                             ctypes.POINTER(i64), ctypes.POINTER(_Frag), i64,
                                             ctypes.POINTER(i64)]
        so.zero_state_init.argtypes = [ctypes.POINTER(_State), ctypes.c_double]
        so.zero_workspace_bytes.argtypes = [i64, i64]
        so.zero_workspace_bytes.restype = ctypes.c_size_t
        so.zero_accumulate_grads.argtypes = [vp, ctypes.POINTER(vp), i32, i32, i64, i32, vp]
        so.zero_accumulate_grads_norm.argtypes = [vp, ctypes.POINTER(vp), i32, i32, i64, i32, vp, i32, vp,
                                                  ctypes.c_size_t, vp]
        so.zero_grad_norm_overflow.argtypes = [ctypes.POINTER(_TList), vp, i32, vp,
                                               ctypes.c_size_t, vp]
        so.zero_adam_step.argtypes = [ctypes.POINTER(_TList)] * 5 + [
            ctypes.POINTER(_HParams), vp, vp, ctypes.c_size_t, vp]
        so.zero_step.argtypes = so.zero_adam_step.argtypes
        so.zero_reduce_grads.argtypes = [ctypes.POINTER(vp), i32, i32, i64, vp, i32, vp, i32, vp,
                                         ctypes.c_size_t, vp]
        so.zero_workspace_stalls.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        for f in ("zero_partition_layout", "zero_state_init", "zero_accumulate_grads", "zero_workspace_stalls",
                  "zero_accumulate_grads_norm", "zero_grad_norm_overflow", "zero_adam_step", "zero_step",
                  "zero_reduce_grads"):
            getattr(so, f).restype = ctypes.c_int
        _lib = so
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != ZERO_OK:
        raise ZeroError(rc, where)


def zero_strerror(code: int) -> str:
    return lib().zero_strerror(int(code)).decode()


# ------------------------------------------------------------------ layout

@dataclass
class Layout:
    shard_numel: int
    padded_total: int
    tensor_offset: np.ndarray  # int64 [n_tensors]
    frags: np.ndarray          # int64 [n_frags, 5]: tensor, tensor_offset, rank, shard_offset, length


def zero_partition_layout(numel: Sequence[int], nd: int, align: int = 128) -> Layout:
    """The flat partition of the tensor list over nd ranks (host only)."""
    n = len(numel)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    offs = (ctypes.c_int64 * max(n, 1))()
    shard, padded, nfr = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = lib().zero_partition_layout(arr, n, int(nd), int(align), ctypes.byref(shard),
                                     ctypes.byref(padded), offs, None, 0, ctypes.byref(nfr))
    if rc not in (ZERO_OK, -6):
        _check(rc, "zero_partition_layout")
    cap = nfr.value
    frags = (_Frag * max(cap, 1))()
    rc = lib().zero_partition_layout(arr, n, int(nd), int(align), ctypes.byref(shard),
                                     ctypes.byref(padded), offs, frags, cap, ctypes.byref(nfr))
    _check(rc, "zero_partition_layout")
    fr = np.frombuffer(frags, dtype=np.int64, count=5 * cap).reshape(cap, 5).copy()
    return Layout(shard.value, padded.value, np.frombuffer(offs, np.int64, count=n).copy(), fr)


# ------------------------------------------------------------------ state, workspace

def zero_state_init(initial_loss_scale: float) -> bytes:
    """The 64-byte initial state (host bytes) for a fresh optimizer."""
    st = _State()
    _check(lib().zero_state_init(ctypes.byref(st), float(initial_loss_scale)), "zero_state_init")
    return ctypes.string_at(ctypes.byref(st), STATE_BYTES)


def new_state(initial_loss_scale: float, device="cuda"):
    """A device uint8[64] tensor holding zero_state_init's state."""
    import torch
    host = torch.frombuffer(bytearray(zero_state_init(initial_loss_scale)), dtype=torch.uint8)
    return host.to(device)


def parse_state(buf) -> dict:
    """Decodes a zero_state_t from 64 host bytes (or a tensor holding them)."""
    if hasattr(buf, "cpu"):
        buf = bytes(buf.cpu().numpy().tobytes())
    st = _State.from_buffer_copy(buf)
    return {name: getattr(st, name) for name, _ in _State._fields_}


def zero_workspace_bytes(max_tensors: int, max_total_numel: int) -> int:
    return int(lib().zero_workspace_bytes(int(max_tensors), int(max_total_numel)))


def new_workspace(max_tensors: int, max_total_numel: int, device="cuda"):
    """A zero-filled device workspace of zero_workspace_bytes() bytes."""
    import torch
    return torch.zeros(zero_workspace_bytes(max_tensors, max_total_numel), dtype=torch.uint8,
                       device=device)


def zero_workspace_stalls(ws, stream=None) -> int:
    """Waits that gave up in calls on this workspace (0 in a healthy run);
    waits for `stream` (default: the current stream) to reach the read."""
    out = ctypes.c_uint32()
    rc = lib().zero_workspace_stalls(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(out),
                                     _stream_ptr(stream, ws.device))
    _check(rc, "zero_workspace_stalls")
    return int(out.value)


# ------------------------------------------------------------------ marshalling

def _dtype_code(t) -> int:
    import torch
    m = {torch.float16: ZERO_F16, torch.bfloat16: ZERO_BF16, torch.float32: ZERO_F32}
    if t.dtype not in m:
        raise TypeError(f"unsupported element type {t.dtype}")
    return m[t.dtype]


def _device_tensor(t, what: str, allow_pinned: bool = False):
    if not t.is_cuda and not (allow_pinned and t.is_pinned()):
        raise ValueError(f"{what} must be a CUDA tensor" +
                         (" or a pinned host tensor" if allow_pinned else ""))
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t


class _ListArgs:
    """Keeps the ctypes arrays of one zero_tlist_t alive for the call."""

    def __new__(cls, tensors, what: str, allow_pinned: bool = False):
        if isinstance(tensors, TensorList):
            return tensors._args
        return super().__new__(cls)

    def __init__(self, tensors, what: str, allow_pinned: bool = False):
        if isinstance(tensors, TensorList):
            return
        if not isinstance(tensors, (list, tuple)):
            tensors = [tensors]
        for t in tensors:
            _device_tensor(t, what, allow_pinned)
        codes = {_dtype_code(t) for t in tensors}
        if len(codes) > 1:
            raise TypeError(f"{what}: mixed element types in one list")
        n = len(tensors)
        self.ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in tensors])
        self.numel = (ctypes.c_int64 * max(n, 1))(*[t.numel() for t in tensors])
        self.tl = _TList(self.ptrs, self.numel, n, codes.pop() if codes else ZERO_F32)
        self.device = tensors[0].device if n else None


class TensorList:
    """A list of device tensors marshalled once into a zero_tlist_t.

    Pass it wherever a list of tensors is accepted; long lists (thousands of
    unflattened tensors) then cost no per-call Python work.  The tensors are
    referenced, so their storage stays alive while the TensorList does."""

    def __init__(self, tensors, what: str = "tensors", allow_pinned: bool = False):
        self.tensors = list(tensors)
        self._args = _ListArgs(self.tensors, what, allow_pinned)

    def __len__(self):
        return len(self.tensors)


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class HParams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_norm: float = 0.0
    min_scale: float = 1.0
    scale_window: int = 1000

    def _c(self) -> _HParams:
        return _HParams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                        self.max_norm, self.min_scale, int(self.scale_window))


# ------------------------------------------------------------------ device calls

def zero_accumulate_grads(acc, grads, overwrite: bool, stream=None) -> None:
    """acc (=|+=) grads[0] + grads[1] + ... (binary32, micro-batch order)."""
    _device_tensor(acc, "acc")
    grads = list(grads)
    for g in grads:
        _device_tensor(g, "grad")
        if g.numel() != acc.numel():
            raise ValueError("micro-batch gradient and accumulator sizes differ")
    codes = {_dtype_code(g) for g in grads}
    if len(codes) != 1:
        raise TypeError("micro-batch gradients must share one element type")
    ptrs = (ctypes.c_void_p * len(grads))(*[g.data_ptr() for g in grads])
    rc = lib().zero_accumulate_grads(ctypes.c_void_p(acc.data_ptr()), ptrs, len(grads),
                                     codes.pop(), acc.numel(), int(bool(overwrite)),
                                     _stream_ptr(stream, acc.device))
    _check(rc, "zero_accumulate_grads")


def zero_accumulate_grads_norm(acc, grads, state, ws, overwrite: bool, accumulate: bool = False,
                               stream=None) -> None:
    """zero_accumulate_grads, then pass 1 (the squared norm and overflow of
    the stored sums into ``state``), in one pass over the micro-batches."""
    _device_tensor(acc, "acc")
    if _dtype_code(acc) != ZERO_F32:
        raise TypeError("acc must be float32")
    grads = list(grads)
    for g in grads:
        _device_tensor(g, "grad")
        if g.numel() != acc.numel():
            raise ValueError("micro-batch gradient and accumulator sizes differ")
    codes = {_dtype_code(g) for g in grads}
    if len(codes) != 1:
        raise TypeError("micro-batch gradients must share one element type")
    _device_tensor(state, "state")
    _device_tensor(ws, "workspace")
    ptrs = (ctypes.c_void_p * len(grads))(*[g.data_ptr() for g in grads])
    rc = lib().zero_accumulate_grads_norm(ctypes.c_void_p(acc.data_ptr()), ptrs, len(grads), codes.pop(),
                                          acc.numel(), int(bool(overwrite)), ctypes.c_void_p(state.data_ptr()),
                                          int(bool(accumulate)), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                          _stream_ptr(stream, acc.device))
    _check(rc, "zero_accumulate_grads_norm")


def zero_reduce_grads(replicas, out, state, ws, accumulate: bool = False, stream=None) -> None:
    """ZeRO stage 2 on one rank: out = mean of the replicas' slices (rank
    order, one division, rounded to out's type), with pass 1 over out."""
    replicas = list(replicas)
    if not 1 <= len(replicas) <= 64:
        raise ValueError("1 to 64 replicas")
    for r in replicas:
        _device_tensor(r, "replica")
        if r.numel() != out.numel():
            raise ValueError("replica and output sizes differ")
    _device_tensor(out, "out")
    _device_tensor(state, "state")
    _device_tensor(ws, "workspace")
    codes = {_dtype_code(r) for r in replicas}
    if len(codes) != 1:
        raise TypeError("replicas must share one element type")
    ptrs = (ctypes.c_void_p * len(replicas))(*[r.data_ptr() for r in replicas])
    rc = lib().zero_reduce_grads(ptrs, len(replicas), codes.pop(), out.numel(),
                                 ctypes.c_void_p(out.data_ptr()), _dtype_code(out),
                                 ctypes.c_void_p(state.data_ptr()), int(bool(accumulate)),
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                 _stream_ptr(stream, state.device))
    _check(rc, "zero_reduce_grads")


def zero_grad_norm_overflow(grads, state, ws, accumulate: bool = False, stream=None) -> None:
    """Pass 1 over one array or a list of arrays; results land in ``state``."""
    la = _ListArgs(grads, "grads")
    _device_tensor(state, "state")
    _device_tensor(ws, "workspace")
    rc = lib().zero_grad_norm_overflow(ctypes.byref(la.tl), ctypes.c_void_p(state.data_ptr()),
                                       int(bool(accumulate)), ctypes.c_void_p(ws.data_ptr()),
                                       ws.numel(), _stream_ptr(stream, state.device))
    _check(rc, "zero_grad_norm_overflow")


def zero_adam_step(grads, master, m, v, p_lp, hp: HParams, state, ws, stream=None) -> None:
    """The decision kernel and pass 2 over one shard or a list of arrays."""
    _step_call("zero_adam_step", grads, master, m, v, p_lp, hp, state, ws, stream)


def zero_step(grads, master, m, v, p_lp, hp: HParams, state, ws, stream=None) -> None:
    """Pass 1, the decision kernel and pass 2 of a single-rank step in one call."""
    _step_call("zero_step", grads, master, m, v, p_lp, hp, state, ws, stream)


class _ListPlan(ctypes.Structure):
    _fields_ = [("ws", ctypes.c_void_p), ("ents", ctypes.c_void_p), ("tiles", ctypes.c_void_p),
                ("chunks", ctypes.c_void_p), ("one", ctypes.c_void_p * 5), ("n", ctypes.c_int64),
                ("total", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
                ("gdtype", ctypes.c_int32), ("pdtype", ctypes.c_int32), ("aligned32", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class ListPlan:
    """A list step prepared once (its tables resident in the workspace): see
    zero_list_prepare.  Holds references to the tensors and the workspace."""

    def __init__(self, c_plan, keep):
        self._c = c_plan
        self._keep = keep

    @property
    def n(self) -> int:
        return int(self._c.n)


def _plan_lib():
    so = lib()
    if not getattr(so, "_plan_ready", False):
        vp = ctypes.c_void_p
        so.zero_list_prepare.argtypes = [ctypes.POINTER(_TList)] * 5 + [vp, ctypes.c_size_t,
                                                                         ctypes.POINTER(_ListPlan), vp]
        so.zero_step_prepared.argtypes = [ctypes.POINTER(_ListPlan), ctypes.POINTER(_HParams), vp, vp,
                                          ctypes.c_size_t, vp]
        so.zero_list_prepare.restype = ctypes.c_int
        so.zero_step_prepared.restype = ctypes.c_int
        so._plan_ready = True
    return so


def zero_list_prepare(grads, master, m, v, p_lp, ws, stream=None) -> ListPlan:
    """The tables of a list step copied into ``ws`` once; the returned plan
    runs the step with zero_step_prepared, copying nothing from the host
    (capturable into a CUDA graph)."""
    lg = _ListArgs(grads, "grads")
    lp_ = _ListArgs(master, "master", allow_pinned=True)
    lm, lv = _ListArgs(m, "m", allow_pinned=True), _ListArgs(v, "v", allow_pinned=True)
    ll = _ListArgs(p_lp, "p_lp") if p_lp is not None else None
    _device_tensor(ws, "workspace")
    plan = _ListPlan()
    rc = _plan_lib().zero_list_prepare(ctypes.byref(lg.tl), ctypes.byref(lp_.tl), ctypes.byref(lm.tl),
                                       ctypes.byref(lv.tl), ctypes.byref(ll.tl) if ll else None,
                                       ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(plan),
                                       _stream_ptr(stream, ws.device))
    _check(rc, "zero_list_prepare")
    return ListPlan(plan, (grads, master, m, v, p_lp, ws, lg, lp_, lm, lv, ll))


def zero_step_prepared(plan: ListPlan, hp: HParams, state, ws, stream=None) -> None:
    """zero_step over the prepared lists, from their resident tables."""
    _device_tensor(state, "state")
    _device_tensor(ws, "workspace")
    h = hp._c()
    rc = _plan_lib().zero_step_prepared(ctypes.byref(plan._c), ctypes.byref(h), ctypes.c_void_p(state.data_ptr()),
                                        ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream, state.device))
    _check(rc, "zero_step_prepared")


def _step_call(fn, grads, master, m, v, p_lp, hp, state, ws, stream):
    lg = _ListArgs(grads, "grads")
    lp_ = _ListArgs(master, "master", allow_pinned=True)
    lm, lv = _ListArgs(m, "m", allow_pinned=True), _ListArgs(v, "v", allow_pinned=True)
    ll = _ListArgs(p_lp, "p_lp") if p_lp is not None else None
    _device_tensor(state, "state")
    _device_tensor(ws, "workspace")
    h = hp._c()
    rc = getattr(lib(), fn)(ctypes.byref(lg.tl), ctypes.byref(lp_.tl), ctypes.byref(lm.tl),
                              ctypes.byref(lv.tl), ctypes.byref(ll.tl) if ll else None,
                              ctypes.byref(h), ctypes.c_void_p(state.data_ptr()),
                              ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                              _stream_ptr(stream, state.device))
    _check(rc, fn)


# ------------------------------------------------------------------ stage 3: parameter gather

class _Piece(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int64), ("rank", ctypes.c_int64),
                ("shard_offset", ctypes.c_int64), ("length", ctypes.c_int64),
                ("layer_offset", ctypes.c_int64)]


def _gather_lib():
    so = lib()
    if not getattr(so, "_gather_ready", False):
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        so.zero_gather_workspace_bytes.argtypes = [i64, i32]
        so.zero_gather_workspace_bytes.restype = ctypes.c_size_t
        so.zero_gather_params.argtypes = [ctypes.POINTER(vp), i32, i64, ctypes.POINTER(_TList),
                                          ctypes.POINTER(i64), vp, ctypes.c_size_t, vp]
        so.zero_scatter_params.argtypes = [ctypes.POINTER(_TList), ctypes.POINTER(i64),
                                           ctypes.POINTER(vp), i32, i64, vp, ctypes.c_size_t, vp]
        so.zero_gather_plan.argtypes = [ctypes.POINTER(i64), i64, ctypes.POINTER(i64), i64, i32, i64,
                                        ctypes.POINTER(i64), ctypes.POINTER(_Piece), i64,
                                        ctypes.POINTER(i64), ctypes.POINTER(i64)]
        for f in ("zero_gather_params", "zero_scatter_params", "zero_gather_plan"):
            getattr(so, f).restype = ctypes.c_int
        so._gather_ready = True
    return so


def zero_gather_workspace_bytes(n_tensors: int, nd: int) -> int:
    return int(_gather_lib().zero_gather_workspace_bytes(int(n_tensors), int(nd)))


def _shard_args(shards):
    shards = list(shards)
    if not shards:
        raise ValueError("at least one shard")
    for t in shards:
        _device_tensor(t, "shard")
    if len({t.numel() for t in shards}) != 1:
        raise ValueError("shards must hold the same number of elements")
    ptrs = (ctypes.c_void_p * len(shards))(*[t.data_ptr() for t in shards])
    return shards, ptrs


def _offsets(offsets, n):
    offs = [int(o) for o in offsets]
    if len(offs) != n:
        raise ValueError("one flat offset per tensor")
    return (ctypes.c_int64 * max(n, 1))(*offs)


def zero_gather_params(shards, tensors, tensor_offset, ws, stream=None) -> None:
    """Shards (rank order) -> tensors: tensor i receives flat elements
    [tensor_offset[i], tensor_offset[i] + numel) of the shards' concatenation."""
    shards, ptrs = _shard_args(shards)
    lt = _ListArgs(tensors, "tensors")
    offs = _offsets(tensor_offset, lt.tl.n)
    _device_tensor(ws, "workspace")
    if lt.tl.n and _dtype_code(shards[0]) != lt.tl.dtype:
        raise TypeError("shards and tensors must share one element type")
    rc = _gather_lib().zero_gather_params(ptrs, len(shards), shards[0].numel(), ctypes.byref(lt.tl),
                                          offs, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                          _stream_ptr(stream, ws.device))
    _check(rc, "zero_gather_params")


def zero_scatter_params(tensors, tensor_offset, shards, ws, stream=None) -> None:
    """Tensors -> shards: the inverse of zero_gather_params (padding untouched)."""
    shards, ptrs = _shard_args(shards)
    lt = _ListArgs(tensors, "tensors")
    offs = _offsets(tensor_offset, lt.tl.n)
    _device_tensor(ws, "workspace")
    if lt.tl.n and _dtype_code(shards[0]) != lt.tl.dtype:
        raise TypeError("shards and tensors must share one element type")
    rc = _gather_lib().zero_scatter_params(ctypes.byref(lt.tl), offs, ptrs, len(shards),
                                           shards[0].numel(), ctypes.c_void_p(ws.data_ptr()),
                                           ws.numel(), _stream_ptr(stream, ws.device))
    _check(rc, "zero_scatter_params")


@dataclass
class GatherPlan:
    layer_flat: np.ndarray   # int64 [n_layers + 1]: flat offset of each layer's first element, then the end
    pieces: np.ndarray       # int64 [n_pieces, 5]: layer, rank, shard_offset, length, layer_offset
    max_layer_numel: int


def zero_gather_plan(numel: Sequence[int], layer_first: Sequence[int], nd: int,
                     align: int = 128) -> GatherPlan:
    """The per-layer gather schedule of stage 3 (host only)."""
    n, nl = len(numel), len(layer_first) - 1
    if nl < 0:
        raise ValueError("layer_first needs at least one entry")
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    lf = (ctypes.c_int64 * max(nl + 1, 1))(*[int(x) for x in layer_first])
    flat = (ctypes.c_int64 * max(nl + 1, 1))()
    npc, big = ctypes.c_int64(), ctypes.c_int64()
    so = _gather_lib()
    rc = so.zero_gather_plan(arr, n, lf, nl, int(nd), int(align), flat, None, 0, ctypes.byref(npc),
                             ctypes.byref(big))
    if rc not in (ZERO_OK, -6):
        _check(rc, "zero_gather_plan")
    cap = npc.value
    pieces = (_Piece * max(cap, 1))()
    rc = so.zero_gather_plan(arr, n, lf, nl, int(nd), int(align), flat, pieces, cap, ctypes.byref(npc),
                             ctypes.byref(big))
    _check(rc, "zero_gather_plan")
    pc = np.frombuffer(pieces, dtype=np.int64, count=5 * cap).reshape(cap, 5).copy()
    return GatherPlan(np.frombuffer(flat, np.int64, count=nl + 1).copy(), pc, big.value)


# ------------------------------------------------------------------ 1-bit Adam

def _onebit_lib():
    so = lib()
    if not getattr(so, "_onebit_ready", False):
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        so.zero_onebit_worker.argtypes = [vp, i32, vp, vp, vp, i64, vp, i64, vp, vp, ctypes.POINTER(_HParams),
                                          i64, vp, vp, ctypes.c_size_t, vp]
        so.zero_onebit_server.argtypes = [ctypes.POINTER(vp), vp, i32, i64, vp, vp, vp, vp, ctypes.c_size_t,
                                          vp]
        so.zero_onebit_update.argtypes = [vp, vp, i32, i64, i64, vp, vp, vp, vp, i32, vp, ctypes.c_size_t,
                                          vp]
        for f in ("zero_onebit_worker", "zero_onebit_server", "zero_onebit_update"):
            getattr(so, f).restype = ctypes.c_int
        so._onebit_ready = True
    return so


def _words_tensor(t, what: str, n_words: int | None = None):
    """A device int32 tensor used as packed sign words."""
    import torch
    _device_tensor(t, what)
    if t.dtype != torch.int32:
        raise TypeError(f"{what} must be an int32 tensor of packed sign words")
    if n_words is not None and t.numel() != n_words:
        raise ValueError(f"{what} must hold {n_words} words")
    return t


def _f32_tensor(t, what: str, n: int | None = None):
    import torch
    _device_tensor(t, what)
    if t.dtype != torch.float32:
        raise TypeError(f"{what} must be float32")
    if n is not None and t.numel() != n:
        raise ValueError(f"{what} must hold {n} elements")
    return t


def zero_onebit_worker(grad, m, x_w, bits, scale, hp: HParams, freeze_step: int, state, ws,
                       stream=None) -> None:
    """1-bit Adam, worker side: the decision (variance frozen at step
    freeze_step), then x = b1*m + (1-b1)*g + e_w compressed to signs (bits,
    int32[n/32]) and one scale (float32[1]).  The error e_w is held in
    deferred form: x_w (float32[n]) and scale hold the previous
    compression's input and scale on entry (e_w = x_w - scale*sign(x_w);
    zeros to start) and this one's on return.  m is the dense momentum
    (float32[n]) or the compressed one, a tuple (signs int32[n/32], scales
    float32[Nd]) from the previous step's servers."""
    n = grad.numel()
    _device_tensor(grad, "grad")
    _f32_tensor(x_w, "x_w", n), _f32_tensor(scale, "scale", 1)
    _words_tensor(bits, "bits", n // 32)
    _device_tensor(state, "state"), _device_tensor(ws, "workspace")
    if isinstance(m, (tuple, list)):
        mb, ms = m
        _words_tensor(mb, "momentum signs", n // 32), _f32_tensor(ms, "momentum scales")
        if n % ms.numel() != 0:
            raise ValueError("momentum scales must split n into equal chunks")
        dense, mbp, msp, chunk = None, ctypes.c_void_p(mb.data_ptr()), ctypes.c_void_p(ms.data_ptr()), n // ms.numel()
    else:
        _f32_tensor(m, "m", n)
        dense, mbp, msp, chunk = ctypes.c_void_p(m.data_ptr()), None, None, 0
    h = hp._c()
    rc = _onebit_lib().zero_onebit_worker(
        ctypes.c_void_p(grad.data_ptr()), _dtype_code(grad), dense, mbp, msp, chunk,
        ctypes.c_void_p(x_w.data_ptr()), n, ctypes.c_void_p(bits.data_ptr()),
        ctypes.c_void_p(scale.data_ptr()), ctypes.byref(h), int(freeze_step),
        ctypes.c_void_p(state.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream_ptr(stream, state.device))
    _check(rc, "zero_onebit_worker")


def zero_onebit_server(worker_bits, worker_scales, x_s, bits, scale, ws, stream=None) -> None:
    """1-bit Adam, server side for this rank's chunk of S = x_s.numel()
    elements: worker_bits (Nd int32 tensors of S/32 words, rank order) and
    worker_scales (float32[Nd]) averaged, plus the server error e_s,
    compressed again.  e_s in deferred form as in zero_onebit_worker: x_s
    and scale (float32[1]) hold the previous server compression's input and
    scale on entry and this one's on return."""
    S = x_s.numel()
    wb = [_words_tensor(b, "worker bits", S // 32) for b in worker_bits]
    _f32_tensor(worker_scales, "worker_scales", len(wb)), _f32_tensor(x_s, "x_s")
    _words_tensor(bits, "bits", S // 32), _f32_tensor(scale, "scale", 1), _device_tensor(ws, "workspace")
    ptrs = (ctypes.c_void_p * max(len(wb), 1))(*[b.data_ptr() for b in wb])
    rc = _onebit_lib().zero_onebit_server(
        ptrs, ctypes.c_void_p(worker_scales.data_ptr()), len(wb), S, ctypes.c_void_p(x_s.data_ptr()),
        ctypes.c_void_p(bits.data_ptr()), ctypes.c_void_p(scale.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream, ws.device))
    _check(rc, "zero_onebit_server")


def zero_onebit_update(bits, server_scales, S: int, numel: int, p, m, v, p_lp, ws, stream=None) -> None:
    """1-bit Adam, every worker: m = the servers' signs times their scales
    (chunk j of S elements from server j), and p updated with the frozen v,
    for the first numel elements; p_lp (fp16/bf16) follows p if given; m may
    be None (the momentum then lives on in its compressed form only)."""
    nd = server_scales.numel()
    _words_tensor(bits, "bits", nd * S // 32), _f32_tensor(server_scales, "server_scales")
    for t, name in ((p, "p"), (v, "v")):
        _f32_tensor(t, name)
        if t.numel() < numel:
            raise ValueError(f"{name} holds fewer than numel elements")
    if m is not None:
        _f32_tensor(m, "m", nd * S)
    lp, code = None, ZERO_F16
    if p_lp is not None:
        _device_tensor(p_lp, "p_lp")
        lp, code = ctypes.c_void_p(p_lp.data_ptr()), _dtype_code(p_lp)
    _device_tensor(ws, "workspace")
    rc = _onebit_lib().zero_onebit_update(
        ctypes.c_void_p(bits.data_ptr()), ctypes.c_void_p(server_scales.data_ptr()), nd, int(S), int(numel),
        ctypes.c_void_p(p.data_ptr()), None if m is None else ctypes.c_void_p(m.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), lp, code,
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream, ws.device))
    _check(rc, "zero_onebit_update")


# ------------------------------------------------------------------ offload (host)

class OffloadScalars(ctypes.Structure):
    """zero_offload_scalars_t: the binary32 scalars of one step's update."""
    _fields_ = [("inv_scale", ctypes.c_float), ("clip", ctypes.c_float),
                ("beta1", ctypes.c_float), ("one_minus_beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("one_minus_beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("step_size", ctypes.c_float),
                ("inv_sqrt_bc2", ctypes.c_float), ("lr_wd", ctypes.c_float),
                ("skip", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _offload_lib():
    so = lib()
    if not getattr(so, "_offload_ready", False):
        vp = ctypes.c_void_p
        so.zero_offload_decide.argtypes = [vp, ctypes.POINTER(_HParams), ctypes.POINTER(OffloadScalars)]
        so.zero_offload_apply.argtypes = [vp, ctypes.c_int32, vp, vp, vp, vp, ctypes.c_int32,
                                          ctypes.c_int64, ctypes.POINTER(OffloadScalars),
                                          ctypes.c_int32]
        so.zero_offload_copy.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int32]
        for f in ("zero_offload_decide", "zero_offload_apply", "zero_offload_copy"):
            getattr(so, f).restype = ctypes.c_int
        so._offload_ready = True
    return so


def _host_array(x, what, code=None):
    """(pointer, element count, dtype code) of a host numpy array or CPU
    tensor; 16-bit patterns stored as uint16 need an explicit code."""
    if hasattr(x, "data_ptr"):
        if x.is_cuda:
            raise ValueError(f"{what} must be in host memory")
        if not x.is_contiguous():
            raise ValueError(f"{what} must be contiguous")
        return x.data_ptr(), x.numel(), _dtype_code(x) if code is None else code
    if not isinstance(x, np.ndarray) or not x.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{what} must be a contiguous numpy array or CPU tensor")
    if code is None:
        code = {np.dtype(np.float16): ZERO_F16, np.dtype(np.float32): ZERO_F32}.get(x.dtype)
        if code is None:
            raise TypeError(f"{what}: pass dtype for {x.dtype} arrays")
    return x.ctypes.data, x.size, code


def default_host_threads() -> int:
    import os
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def zero_offload_decide(host_state, hp: HParams) -> OffloadScalars:
    """The step decision on a 64-byte host zero_state_t (numpy uint8 array or
    CPU uint8 tensor), updated in place; returns the element scalars."""
    ptr, n, _ = _host_array(host_state, "host_state", code=-1)
    if n != STATE_BYTES:
        raise ValueError("host_state must hold the 64 bytes of a zero_state_t")
    out = OffloadScalars()
    h = hp._c()
    _check(_offload_lib().zero_offload_decide(ctypes.c_void_p(ptr), ctypes.byref(h),
                                               ctypes.byref(out)), "zero_offload_decide")
    return out


def zero_offload_apply(grad, master, m, v, p_lp, scalars: OffloadScalars, gdtype=None,
                       pdtype=None, n_threads: int = 0) -> None:
    """The element update on host arrays (numpy or CPU tensors); gdtype /
    pdtype: "f16", "bf16" or "f32" where the array type does not say it."""
    codes = {"f16": ZERO_F16, "bf16": ZERO_BF16, "f32": ZERO_F32, None: None}
    gp, n, gc = _host_array(grad, "grad", codes[gdtype])
    arrs = []
    for a, name in ((master, "master"), (m, "m"), (v, "v")):
        ptr, na, code = _host_array(a, name)
        if code != ZERO_F32:
            raise TypeError(f"{name} must be float32")
        if na != n:
            raise ValueError("array sizes differ")
        arrs.append(ptr)
    lp, lc = None, ZERO_F16
    if p_lp is not None:
        lptr, ln, lc = _host_array(p_lp, "p_lp", codes[pdtype])
        if ln != n:
            raise ValueError("array sizes differ")
        lp = ctypes.c_void_p(lptr)
    rc = _offload_lib().zero_offload_apply(
        ctypes.c_void_p(gp), gc, ctypes.c_void_p(arrs[0]), ctypes.c_void_p(arrs[1]),
        ctypes.c_void_p(arrs[2]), lp, lc, n, ctypes.byref(scalars),
        n_threads or default_host_threads())
    _check(rc, "zero_offload_apply")


def zero_offload_copy(dst, src, n_threads: int = 0) -> None:
    """Multi-threaded host memcpy between equally sized host buffers."""
    dp, dn, _ = _host_array(dst, "dst", code=-1)
    sp, sn, _ = _host_array(src, "src", code=-1)
    nbytes = (dst.nbytes if isinstance(dst, np.ndarray) else dst.numel() * dst.element_size())
    sbytes = (src.nbytes if isinstance(src, np.ndarray) else src.numel() * src.element_size())
    if nbytes != sbytes:
        raise ValueError("buffer sizes differ")
    _check(_offload_lib().zero_offload_copy(ctypes.c_void_p(dp), ctypes.c_void_p(sp), nbytes,
                                             n_threads or default_host_threads()),
           "zero_offload_copy")
