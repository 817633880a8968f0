"""The oracle: TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.

A plain, slow CPU statement of what one ZeRO data-parallel rank computes in
its mixed-precision optimizer step, used to prove the CUDA library right.
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import it.  It shares no code with the CUDA library (neither imports
the other); the two meet only through the seeded synthetic inputs of
``zero_synth``.

Parts:
  * ``zero_oracle.c`` -- the per-element arithmetic (accumulate, unscale +
    overflow + squared norm, the step decision, clip + AdamW + cast), scalar C
    in binary32 as the pages' fp32 state fixes it; wrapped here with ctypes.
  * ``partition_layout`` -- the flat, padded partition of the model states over
    Nd ranks, in plain Python integers.
  * ``gather_params`` / ``scatter_params`` / ``gather_plan`` -- stage 3: the
    inverse layout (shards back to tensors) and its per-layer schedule.
  * ``model_state_bytes`` / ``comm_volume`` -- the pages' memory and
    communication arithmetic.
  * ``onebit_*`` -- 1-bit Adam's compression stage (worker compression with
    error feedback, the server's average and recompression, the update with
    the frozen variance), element arithmetic in ``zero_oracle.c``.

Sources: "ZeRO: Memory Optimizations Toward Training Trillion Parameter
Models - 中文验证版" (ai-papers.xuzou.cn/zh/papers/zero_2019/), cited as
[ZeRO card §section]; "探秘微软大规模人工智能的新框架 ZeRO-2" (infoq.cn), cited
as [ZeRO-2]; DeepSpeed release news (lxsoso.com/blog/19320.html), cited as
[DS news].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_LIB = os.path.join(_HERE, "libzero_oracle.so")

DTYPES = {"f16": 0, "bf16": 1, "f32": 2}


def build(force: bool = False) -> str:
    """Compiles the C oracle with gcc: -O2, binary32 evaluated as written
    (no FMA contraction, no fast-math), single-threaded."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
             "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("max_norm", ctypes.c_double),
                ("min_scale", ctypes.c_double), ("scale_window", ctypes.c_int64)]


class _Scaler(ctypes.Structure):
    _fields_ = [("loss_scale", ctypes.c_double), ("step", ctypes.c_int64),
                ("good_steps", ctypes.c_int64)]


class _Step(ctypes.Structure):
    _fields_ = [("inv_scale", ctypes.c_float), ("clip", ctypes.c_float),
                ("beta1", ctypes.c_float), ("one_minus_beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("one_minus_beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("step_size", ctypes.c_float),
                ("inv_sqrt_bc2", ctypes.c_float), ("lr_wd", ctypes.c_float),
                ("skip", ctypes.c_int32), ("norm", ctypes.c_double)]


_lib = None


def load(path: str):
    """Opens a built oracle library and declares its C signatures."""
    so = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    so.zo_f32_to_lp.argtypes = [vp, vp, ctypes.c_int, i64]
    so.zo_lp_to_f32.argtypes = [vp, ctypes.c_int, vp, i64]
    so.zo_accumulate.argtypes = [vp, ctypes.POINTER(vp), i32, ctypes.c_int, i64, i32]
    so.zo_norm_overflow.argtypes = [vp, ctypes.c_int, i64, ctypes.c_float,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32)]
    so.zo_decide.argtypes = [ctypes.POINTER(_HParams), ctypes.POINTER(_Scaler),
                             ctypes.c_double, i32, ctypes.POINTER(_Step)]
    so.zo_adam_apply.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, ctypes.c_int, i64,
                                 ctypes.POINTER(_Step)]
    so.zo_adam_apply_sampled.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                         ctypes.c_int, i64, ctypes.POINTER(_Step)]
    so.zo_reduce_mean.argtypes = [ctypes.POINTER(vp), i32, ctypes.c_int, i64, vp, ctypes.c_int]
    f32 = ctypes.c_float
    so.zo_onebit_worker.argtypes = [vp, ctypes.c_int, i64, ctypes.POINTER(_Step), vp, vp, vp,
                                    ctypes.POINTER(f32), f32, vp]
    so.zo_onebit_server.argtypes = [ctypes.POINTER(vp), vp, i32, i64, vp, vp, ctypes.POINTER(f32),
                                    f32, i32, vp]
    so.zo_onebit_update.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp, ctypes.c_int,
                                    ctypes.POINTER(_Step)]
    for f in ("zo_f32_to_lp", "zo_lp_to_f32", "zo_accumulate", "zo_norm_overflow",
              "zo_decide", "zo_adam_apply", "zo_adam_apply_sampled", "zo_reduce_mean",
              "zo_onebit_worker", "zo_onebit_server", "zo_onebit_update"):
        getattr(so, f).restype = None
    return so


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def compile_source(src_path: str, out_path: str) -> str:
    """Builds another copy of the oracle source (same flags); the mutation
    test uses it to check that the pins catch planted mistakes."""
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-w",
         "-shared", "-fPIC", "-o", out_path, src_path, "-lm"])
    return out_path


# ---------------------------------------------------------------- helpers

def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """The raw element array the C side reads: uint16 bit patterns for the
    16-bit types (numpy float16 arrays are accepted as they are), float32."""
    if dtype == "f32":
        assert a.dtype == np.float32
        return a
    if a.dtype == np.float16:
        assert dtype == "f16"
        return a.view(np.uint16)
    assert a.dtype == np.uint16
    return a


def to_lp(x: np.ndarray, dtype: str) -> np.ndarray:
    """binary32 -> binary16 / bfloat16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().zo_f32_to_lp(_ptr(x), _ptr(out), DTYPES[dtype], x.size)
    return out


def from_lp(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(_bits(bits, dtype))
    out = np.empty(bits.shape, np.float32)
    lib().zo_lp_to_f32(_ptr(bits), DTYPES[dtype], _ptr(out), bits.size)
    return out


# ---------------------------------------------------------------- hparams

@dataclass
class HParams:
    """AdamW and loss-scaler settings.  Defaults: lr 1e-3, betas (0.9, 0.999),
    eps 1e-8, weight decay 0.01, no clipping, scale floor 1, growth after
    1000 clean steps."""
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
                        self.max_norm, self.min_scale, self.scale_window)


@dataclass
class Scaler:
    loss_scale: float = 1.0
    step: int = 0
    good_steps: int = 0


@dataclass
class Step:
    """The outcome of one step's decision: skip flag, norm and the binary32
    scalars of the element update."""
    skip: bool
    norm: float
    scalars: dict = field(default_factory=dict)
    _c: object = None


# ---------------------------------------------------------------- the step

def accumulate(acc: np.ndarray, bufs: list[np.ndarray], dtype: str, overwrite: bool) -> None:
    """[DS news] gradient accumulation: acc (=|+=) g_0 + g_1 + ... in
    micro-batch order, binary32."""
    arrs = [np.ascontiguousarray(_bits(b, dtype)) for b in bufs]
    assert acc.dtype == np.float32 and all(a.size == acc.size for a in arrs)
    ptrs = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    lib().zo_accumulate(_ptr(acc), ptrs, len(arrs), DTYPES[dtype], acc.size, int(overwrite))


def reduce_mean(bufs: list[np.ndarray], dtype: str, out_dtype: str) -> np.ndarray:
    """ZeRO stage 2's gradient reduction on one shard: the mean over the Nd
    replicas, binary32 sum in rank order, one division, rounded to out_dtype
    (uint16 bit patterns for 16-bit outputs, float32 otherwise)."""
    arrs = [np.ascontiguousarray(_bits(b, dtype)) for b in bufs]
    n = arrs[0].size
    assert all(a.size == n for a in arrs) and len(arrs) >= 1
    out = np.empty(n, np.float32 if out_dtype == "f32" else np.uint16)
    ptrs = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    lib().zo_reduce_mean(ptrs, len(arrs), DTYPES[dtype], n, _ptr(out), DTYPES[out_dtype])
    return out


def norm_overflow(grads: list[np.ndarray], dtype: str, loss_scale: float):
    """Global (sum of g^2, found_inf) of the unscaled gradient over every
    array in ``grads`` taken in order (binary64 sum in index order)."""
    s = ctypes.c_double(0.0)
    bad = ctypes.c_int32(0)
    inv = np.float32(1.0 / loss_scale)
    for g in grads:
        a = np.ascontiguousarray(_bits(g, dtype))
        lib().zo_norm_overflow(_ptr(a), DTYPES[dtype], a.size, ctypes.c_float(inv),
                               ctypes.byref(s), ctypes.byref(bad))
    return s.value, int(bad.value)


def decide(hp: HParams, sc: Scaler, sumsq: float, found_inf: int) -> Step:
    """Skip-or-apply, loss-scale update, step count and step scalars; ``sc``
    is advanced in place."""
    csc = _Scaler(sc.loss_scale, sc.step, sc.good_steps)
    st = _Step()
    lib().zo_decide(ctypes.byref(hp._c()), ctypes.byref(csc), ctypes.c_double(sumsq),
                    int(found_inf), ctypes.byref(st))
    sc.loss_scale, sc.step, sc.good_steps = csc.loss_scale, csc.step, csc.good_steps
    scal = {name: getattr(st, name) for name, _ in _Step._fields_ if name not in ("skip", "norm")}
    return Step(bool(st.skip), st.norm, scal, st)


def with_clip(step: Step, clip: float) -> Step:
    """The same step with another binary32 clip coefficient, for comparing an
    implementation whose norm rounded its clip coefficient the other way."""
    st = _Step()
    ctypes.memmove(ctypes.byref(st), ctypes.byref(step._c), ctypes.sizeof(_Step))
    st.clip = float(np.float32(clip))
    scal = dict(step.scalars)
    scal["clip"] = st.clip
    return Step(step.skip, step.norm, scal, st)


def adam_apply(g: np.ndarray, gdtype: str, p: np.ndarray, m: np.ndarray, v: np.ndarray,
               p_lp: np.ndarray | None, pdtype: str, step: Step) -> None:
    """Clip + AdamW + cast over whole arrays, in place."""
    ga = np.ascontiguousarray(_bits(g, gdtype))
    for a in (p, m, v):
        assert a.dtype == np.float32 and a.size == ga.size and a.flags["C_CONTIGUOUS"]
    lp = None if p_lp is None else _bits(p_lp, pdtype)
    lib().zo_adam_apply(_ptr(ga), DTYPES[gdtype], _ptr(p), _ptr(m), _ptr(v), _ptr(lp),
                        DTYPES[pdtype], ga.size, ctypes.byref(step._c))


def adam_apply_sampled(g: np.ndarray, gdtype: str, idx: np.ndarray, p: np.ndarray,
                       m: np.ndarray, v: np.ndarray, p_lp: np.ndarray | None, pdtype: str,
                       step: Step) -> None:
    """The update for the elements ``idx`` of a full gradient array; the
    state arrays hold those elements only."""
    ga = np.ascontiguousarray(_bits(g, gdtype))
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    assert idx.size == 0 or (idx.min() >= 0 and idx.max() < ga.size)
    for a in (p, m, v):
        assert a.dtype == np.float32 and a.size == idx.size
    lp = None if p_lp is None else _bits(p_lp, pdtype)
    lib().zo_adam_apply_sampled(_ptr(ga), DTYPES[gdtype], _ptr(idx), _ptr(p), _ptr(m), _ptr(v),
                                _ptr(lp), DTYPES[pdtype], idx.size, ctypes.byref(step._c))


def adam_step(grads: list[np.ndarray], gdtype: str, p: list[np.ndarray], m: list[np.ndarray],
              v: list[np.ndarray], p_lp: list[np.ndarray | None], pdtype: str, hp: HParams,
              sc: Scaler) -> Step:
    """One full step over one rank's shard, or over every rank's shard in rank
    order: the global norm and overflow first, then the decision, then the
    element update of every array."""
    sumsq, bad = norm_overflow(grads, gdtype, sc.loss_scale)
    st = decide(hp, sc, sumsq, bad)
    for i, g in enumerate(grads):
        adam_apply(g, gdtype, p[i], m[i], v[i], p_lp[i], pdtype, st)
    return st


# ---------------------------------------------------------------- 1-bit Adam

def frozen_variance(step: Step, hp: HParams, t_freeze: int) -> Step:
    """1-bit Adam's compression stage: the step with the variance's bias
    correction frozen at the last warm-up step T_w, 1/sqrt(1 - b2^T_w)
    (binary64, rounded once), since the variance itself stays frozen."""
    import math
    st = _Step()
    ctypes.memmove(ctypes.byref(st), ctypes.byref(step._c), ctypes.sizeof(_Step))
    if not step.skip:
        st.inv_sqrt_bc2 = float(np.float32(1.0 / math.sqrt(1.0 - hp.beta2 ** float(t_freeze))))
    scal = dict(step.scalars)
    scal["inv_sqrt_bc2"] = st.inv_sqrt_bc2
    return Step(step.skip, step.norm, scal, st)


def _words(n: int) -> int:
    return (n + 31) // 32


def _x_out(x_out: np.ndarray | None, n: int):
    if x_out is None:
        return None
    assert x_out.dtype == np.float32 and x_out.size == n and x_out.flags["C_CONTIGUOUS"]
    return _ptr(x_out)


def onebit_worker(g: np.ndarray, gdtype: str, step: Step, m: np.ndarray, e: np.ndarray,
                  scale: float | None = None, x_out: np.ndarray | None = None):
    """Worker side of 1-bit Adam's compressed all-reduce: local momentum
    b1*m + (1-b1)*g, plus the worker error e, compressed to signs and one
    scale; e (float32) is updated in place, m is read only.  Returns (bits
    uint32[n/32], scale); unchanged inputs and (None, None) on a skipped
    step.  ``scale`` forces the scale (see onebit_compress in the C file);
    ``x_out`` (float32[n]) receives the compressed value x itself."""
    ga = np.ascontiguousarray(_bits(g, gdtype))
    n = ga.size
    assert m.dtype == np.float32 and e.dtype == np.float32 and m.size == n == e.size
    bits = np.zeros(_words(n), np.uint32)
    out = ctypes.c_float(0.0)
    lib().zo_onebit_worker(_ptr(ga), DTYPES[gdtype], n, ctypes.byref(step._c), _ptr(m), _ptr(e),
                           _ptr(bits), ctypes.byref(out), -1.0 if scale is None else float(scale),
                           _x_out(x_out, n))
    return (None, None) if step.skip else (bits, out.value)


def onebit_server(bits: list[np.ndarray], scales: list[float], f: np.ndarray,
                  scale: float | None = None, skip: bool = False, x_out: np.ndarray | None = None):
    """Server side for one chunk of S elements: the Nd workers' signs on the
    chunk (uint32[S/32] each, rank order) and scales, averaged, plus the
    server error f (float32[S], updated in place), compressed again.
    Returns (bits uint32[S/32], scale); ``x_out`` (float32[S]) receives
    the compressed value itself."""
    S = f.size
    arrs = [np.ascontiguousarray(b, dtype=np.uint32) for b in bits]
    assert all(a.size == _words(S) for a in arrs) and f.dtype == np.float32
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    ptrs = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    out_bits = np.zeros(_words(S), np.uint32)
    out = ctypes.c_float(0.0)
    lib().zo_onebit_server(ptrs, _ptr(sc), len(arrs), S, _ptr(f), _ptr(out_bits), ctypes.byref(out),
                           -1.0 if scale is None else float(scale), int(skip), _x_out(x_out, S))
    return (None, None) if skip else (out_bits, out.value)


def onebit_update(bits: np.ndarray, scales: list[float], S: int, numel: int, p: np.ndarray,
                  m: np.ndarray, v: np.ndarray, p_lp: np.ndarray | None, pdtype: str,
                  step: Step) -> None:
    """Every worker: the synchronised momentum (the servers' signs, chunk j
    scaled by scales[j]) into m over the whole padded buffer of
    len(scales) * S elements, and the update of p with the frozen variance
    v for the first ``numel`` elements; in place."""
    b = np.ascontiguousarray(bits, dtype=np.uint32)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    n = sc.size * S
    assert b.size * 32 >= n and numel <= n
    assert m.dtype == np.float32 and m.size >= n and m.flags["C_CONTIGUOUS"]
    for a in (p, v):
        assert a.dtype == np.float32 and a.size >= numel and a.flags["C_CONTIGUOUS"]
    lp = None if p_lp is None else _bits(p_lp, pdtype)
    lib().zo_onebit_update(_ptr(b), _ptr(sc), S, n, numel, _ptr(p), _ptr(m), _ptr(v), _ptr(lp),
                           DTYPES[pdtype], ctypes.byref(step._c))


@dataclass
class OnebitResult:
    step: Step
    worker_bits: list = field(default_factory=list)
    worker_scales: list = field(default_factory=list)
    server_bits: list = field(default_factory=list)
    server_scales: list = field(default_factory=list)
    worker_x: list = field(default_factory=list)   # each compression's input x
    server_x: list = field(default_factory=list)


def onebit_step(grads: list[np.ndarray], gdtype: str, S: int, numel: int, p: np.ndarray,
                m: np.ndarray, v: np.ndarray, e_w: list[np.ndarray], e_s: list[np.ndarray],
                p_lp: np.ndarray | None, pdtype: str, hp: HParams, sc: Scaler, t_freeze: int,
                worker_scales: list | None = None, server_scales: list | None = None,
                clip: float | None = None) -> OnebitResult:
    """One compression-stage step of 1-bit Adam over all Nd = len(grads)
    workers (every worker holds the same p, m, v; its own gradient and error
    e_w[i]; rank j serves chunk j with error e_s[j]).  The overflow flag and
    the squared norm are summed over the workers' gradients.  Optional
    worker_scales / server_scales force the scales (another implementation's
    rounding of the norms); ``clip`` likewise forces the binary32 clip
    coefficient (see with_clip)."""
    nd = len(grads)
    assert p.size == nd * S
    sumsq, bad = norm_overflow(grads, gdtype, sc.loss_scale)
    st = decide(hp, sc, sumsq, bad)
    if clip is not None and not st.skip:
        st = with_clip(st, clip)
    st = frozen_variance(st, hp, t_freeze)
    res = OnebitResult(st)
    if st.skip:
        return res
    for i in range(nd):
        x = np.empty(nd * S, np.float32)
        b, s_ = onebit_worker(grads[i], gdtype, st, m, e_w[i],
                              None if worker_scales is None else worker_scales[i], x_out=x)
        res.worker_bits.append(b)
        res.worker_scales.append(s_)
        res.worker_x.append(x)
    w = S // 32
    for j in range(nd):
        x = np.empty(S, np.float32)
        b, s_ = onebit_server([res.worker_bits[i][j * w:(j + 1) * w] for i in range(nd)],
                              res.worker_scales, e_s[j],
                              None if server_scales is None else server_scales[j], x_out=x)
        res.server_bits.append(b)
        res.server_scales.append(s_)
        res.server_x.append(x)
    onebit_update(np.concatenate(res.server_bits), res.server_scales, S, numel, p, m, v, p_lp,
                  pdtype, st)
    return res


def onebit_comm_ratio(warmup_fraction: float, full_bits: int = 32) -> float:
    """Communication of plain data-parallel Adam over 1-bit Adam's, per
    element and step: the warm-up steps send full-precision values, the rest
    one bit (the scales are negligible)."""
    return full_bits / (warmup_fraction * full_bits + (1.0 - warmup_fraction))


# ---------------------------------------------------------------- layout

@dataclass
class Layout:
    shard_numel: int
    padded_total: int
    tensor_offset: list[int]
    # (tensor index, offset in tensor, rank, offset in shard, length)
    frags: list[tuple[int, int, int, int, int]]


def partition_layout(numel: list[int], nd: int, align: int) -> Layout:
    """[ZeRO card §方法适配]: the model states are split over the Nd
    data-parallel ranks instead of replicated.  Reading: the tensors are
    concatenated in list order into one flat buffer, the flat length is padded
    at the tail up to a multiple of nd * align, and rank r owns the contiguous
    shard [r*S, (r+1)*S) with S = ceil(total / (nd*align)) * align.  A tensor
    that straddles a shard boundary is cut there; each piece is one fragment."""
    if nd <= 0 or align <= 0:
        raise ValueError("nd and align must be positive")
    total = 0
    offsets = []
    for n in numel:
        if n < 0:
            raise ValueError("negative numel")
        offsets.append(total)
        total += n
    unit = nd * align
    shard = -(-total // unit) * align
    frags = []
    for t, n in enumerate(numel):
        pos, end = offsets[t], offsets[t] + n
        while pos < end:
            r = pos // shard
            stop = min(end, (r + 1) * shard)
            frags.append((t, pos - offsets[t], r, pos - r * shard, stop - pos))
            pos = stop
    return Layout(shard, nd * shard, offsets, frags)


# ---------------------------------------------------------------- stage 3: parameter gather

def gather_params(shards: list[np.ndarray], tensor_offset: list[int],
                  numel: list[int]) -> list[np.ndarray]:
    """[ZeRO card §方法适配]: stage 3 partitions the parameters themselves, so
    a rank holds only its shard and must assemble a tensor from the ranks'
    shards before it is used.  Reading: the flat parameter buffer is the
    concatenation of the Nd shards in rank order (the inverse of
    ``partition_layout``), and tensor i is its slice [offset_i, offset_i +
    numel_i).  Elements are moved unchanged."""
    full = np.concatenate(shards)
    return [full[o:o + n].copy() for o, n in zip(tensor_offset, numel)]


def scatter_params(tensors: list[np.ndarray], tensor_offset: list[int], nd: int,
                   shard_numel: int) -> list[np.ndarray]:
    """The opposite direction of ``gather_params``: the tensors written at
    their flat offsets into a zero flat buffer of nd * S elements, cut into
    the Nd shards [r*S, (r+1)*S) (the padding stays zero)."""
    dtype = tensors[0].dtype if tensors else np.float16
    full = np.zeros(nd * shard_numel, dtype)
    for t, o in zip(tensors, tensor_offset):
        full[o:o + t.size] = t
    return [full[r * shard_numel:(r + 1) * shard_numel].copy() for r in range(nd)]


@dataclass
class LayerGather:
    begin: int                       # flat range of the layer's tensors
    end: int
    pieces: list = field(default_factory=list)  # (rank, shard_offset, length, layer_offset)


def gather_plan(numel: list[int], layer_first: list[int], nd: int, align: int) -> list[LayerGather]:
    """Per-layer gather schedule of stage 3.  [ZeRO card §方法适配]: stage 3
    shards the parameters over the data-parallel ranks; the ZeRO-Infinity
    page's memory-centric tiling works on one layer at a time.  Reading: a
    layer is a run of consecutive tensors (``layer_first`` holds the first
    tensor of each layer and ends with the tensor count), so its parameters
    are one flat range [begin, end); rank r contributes the part of that range
    that lies in its shard [r*S, (r+1)*S), one contiguous piece, placed at the
    same distance from ``begin`` in the gathered layer."""
    lay = partition_layout(numel, nd, align)
    S = lay.shard_numel
    offs = lay.tensor_offset + [sum(numel)]
    plan = []
    for L in range(len(layer_first) - 1):
        lg = LayerGather(offs[layer_first[L]], offs[layer_first[L + 1]])
        begin, end = lg.begin, lg.end
        for r in range(nd):
            lo, hi = max(begin, r * S), min(end, (r + 1) * S)
            if lo < hi:
                lg.pieces.append((r, lo - r * S, hi - lo, lo - begin))
        plan.append(lg)
    return plan


def comm_volume(psi: float, stage: int) -> float:
    """Elements each rank sends per training step (ring collectives, large
    Nd).  [ZeRO card §方法适配]: stages 1 and 2 keep the communication volume
    of data parallelism; stage 3 raises it by about half.  Reading: data
    parallelism all-reduces the gradient (a reduce-scatter plus an all-gather,
    2 psi); stages 1 and 2 do a reduce-scatter of the gradient and an
    all-gather of the updated parameters (2 psi); stage 3 gathers the
    parameters for the forward and again for the backward pass and
    reduce-scatters the gradient (3 psi)."""
    if stage in (0, 1, 2):
        return 2.0 * psi
    if stage == 3:
        return 3.0 * psi
    raise ValueError("stage must be 0..3")


# ---------------------------------------------------------------- memory

BYTES_PER_PARAM = {"p16": 2, "g16": 2, "p32": 4, "m32": 4, "v32": 4}


def model_state_bytes(psi: int, nd: int = 1, stage: int = 0) -> float:
    """Per-rank model-state bytes of mixed-precision Adam.

    [ZeRO card §瓶颈]: fp16 parameter and gradient plus fp32 parameter,
    momentum and variance, i.e. 2 + 2 + 12 = 16 bytes per parameter.
    [ZeRO card §方法适配]: stage 1 partitions the 12 optimizer-state bytes over
    the nd ranks, stage 2 the gradient's 2 bytes as well, stage 3 the
    parameter's 2 bytes too; stage 0 is plain data parallelism (replicated)."""
    b = BYTES_PER_PARAM
    opt = b["p32"] + b["m32"] + b["v32"]
    if stage == 0:
        return psi * (b["p16"] + b["g16"] + opt)
    if stage == 1:
        return psi * (b["p16"] + b["g16"]) + psi * opt / nd
    if stage == 2:
        return psi * b["p16"] + psi * (b["g16"] + opt) / nd
    if stage == 3:
        return psi * (b["p16"] + b["g16"] + opt) / nd
    raise ValueError("stage must be 0..3")
