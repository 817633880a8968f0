"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke
check.  This module holds workload shapes and random draws only: no part of
the optimizer step, the layout or the memory arithmetic lives here, so both
the oracle and the CUDA library can be fed from it without sharing method code.

Workloads (all synthetic; there is no dataset on this path):
  * ``tiny``       -- a 2-layer transformer state, hidden 256, vocab 1024,
                      14 tensors (1,836,288 params), Nd = 1, fp16 gradients of
                      N(0, 1e-3) times loss scale 1024, fp32 master N(0, 0.02).
  * ``gpt2_1p5b``  -- the GPT-2 1.5B tensor list (48 layers, hidden 1600,
                      vocab 50257, 1024 positions; 580 tensors, 1,557,611,200
                      params), the model the ZeRO pages size at 24 GB of state.
  * ``stack_100b`` -- 125 GPT layers of hidden 8192 (1,500 tensors,
                      100,676,608,000 params), the 100B configuration the ZeRO
                      evaluation trains on 400 GPUs (16-way model parallel x
                      25-way data parallel).
  * ``frag_10k``   -- 10,000 tensors with log-normal sizes (median 4096,
                      sigma 2, clipped to [1, 2^24], one forced to 2^24).
  * flat shards of 2^k params for the size sweep.
"""
from __future__ import annotations

import hashlib

import numpy as np

# ------------------------------------------------------------------ shapes

def tiny_transformer_shapes(layers: int = 2, hidden: int = 256, vocab: int = 1024):
    """Per layer: fused qkv [3h, h], attention out [h, h], MLP in [4h, h],
    MLP out [h, 4h], two norm weights [h]; then token embedding [vocab, h]
    and the final norm weight [h]."""
    h = hidden
    shapes = []
    for _ in range(layers):
        shapes += [(3 * h, h), (h, h), (4 * h, h), (h, 4 * h), (h,), (h,)]
    shapes += [(vocab, h), (h,)]
    return shapes


def gpt_layer_shapes(h: int):
    """The 12 tensors of one GPT-2 block in state-dict order: ln_1 (w, b),
    attn.c_attn (w [h, 3h], b), attn.c_proj (w [h, h], b), ln_2 (w, b),
    mlp.c_fc (w [h, 4h], b), mlp.c_proj (w [4h, h], b): 12h^2 + 13h params."""
    return [(h,), (h,), (h, 3 * h), (3 * h,), (h, h), (h,), (h,), (h,),
            (h, 4 * h), (4 * h,), (4 * h, h), (h,)]


def gpt2_shapes(layers: int = 48, hidden: int = 1600, vocab: int = 50257, positions: int = 1024):
    shapes = [(vocab, hidden), (positions, hidden)]
    for _ in range(layers):
        shapes += gpt_layer_shapes(hidden)
    shapes += [(hidden,), (hidden,)]
    return shapes


def gpt2_layer_first(layers: int = 48):
    """Layer boundaries of ``gpt2_shapes`` as first-tensor indices: the two
    embeddings, each block's 12 tensors, the final norm's two, then the
    tensor count."""
    return [0] + [2 + 12 * k for k in range(layers + 1)] + [2 + 12 * layers + 2]


def layer_stack_shapes(layers: int = 125, hidden: int = 8192):
    shapes = []
    for _ in range(layers):
        shapes += gpt_layer_shapes(hidden)
    return shapes


def frag_sizes(n_tensors: int = 10_000, median: int = 4096, sigma: float = 2.0,
               max_numel: int = 1 << 24, seed: int = 0):
    """Log-normal tensor sizes from numpy's default_rng(seed); clipped to
    [1, max_numel]; the first tensor is forced to max_numel."""
    rng = np.random.default_rng(seed)
    x = rng.lognormal(mean=np.log(median), sigma=sigma, size=n_tensors)
    sizes = np.clip(np.rint(x), 1, max_numel).astype(np.int64)
    sizes[0] = max_numel
    return [int(s) for s in sizes]


def numels(shapes):
    out = []
    for s in shapes:
        n = 1
        for d in s:
            n *= d
        out.append(n)
    return out


# ------------------------------------------------------------------ workloads

WORKLOADS = {
    "tiny": dict(numel=lambda: numels(tiny_transformer_shapes()), nd=1, rank=0, align=128,
                 gdtype="f16", pdtype="f16", loss_scale=1024.0, max_norm=0.0, steps=3,
                 micro_batches=1, inf_step=None),
    "gpt2_1p5b_nd16": dict(numel=lambda: numels(gpt2_shapes()), nd=16, rank=0, align=128,
                           gdtype="f16", pdtype="f16", loss_scale=65536.0, max_norm=0.0,
                           steps=5, micro_batches=1, inf_step=2),
    "gpt2_1p5b_full": dict(numel=lambda: numels(gpt2_shapes()), nd=1, rank=0, align=128,
                           gdtype="f16", pdtype="f16", loss_scale=1.0, max_norm=1.0, steps=3,
                           micro_batches=1, inf_step=None),
    "stack_100b_nd400": dict(numel=lambda: numels(layer_stack_shapes()), nd=400, rank=0,
                             align=128, gdtype="bf16", pdtype="bf16", loss_scale=1.0,
                             max_norm=1.0, steps=3, micro_batches=4, inf_step=None),
    "frag_10k": dict(numel=lambda: frag_sizes(), nd=1, rank=0, align=128, gdtype="f16",
                     pdtype="f16", loss_scale=1024.0, max_norm=0.0, steps=3, micro_batches=1,
                     inf_step=None),
}

HPARAMS = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
GRAD_STD = 1e-3
MASTER_STD = 0.02

# ------------------------------------------------------------------ draws

_STREAMS = {"master": 1, "grad": 2, "inf": 3, "sample": 4, "misc": 5}


def stream_seed(seed: int, stream: str, *keys: int) -> int:
    """A 63-bit seed for one named stream of draws (e.g. the gradient of
    step 2, micro-batch 1), stable across machines."""
    h = hashlib.sha256(repr((int(seed), _STREAMS[stream]) + tuple(int(k) for k in keys)).encode())
    return int.from_bytes(h.digest()[:8], "little") >> 1


def host_normal(n: int, std: float, seed: int, stream: str, *keys: int) -> np.ndarray:
    """n draws of N(0, std^2) as float32 from numpy's PCG64 generator."""
    rng = np.random.default_rng(stream_seed(seed, stream, *keys))
    x = rng.standard_normal(n, dtype=np.float32)
    x *= np.float32(std)
    return x


def host_cast(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> the stored element type: np.float16 for 'f16', uint16 bit
    patterns for 'bf16' (torch's CPU cast, round to nearest even), float32."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def host_grad(n: int, seed: int, step: int, scale: float, dtype: str, micro: int = 0,
              std: float = GRAD_STD) -> np.ndarray:
    """The stored gradient of one step (and micro-batch): N(0, std^2) times
    the loss scale in force, cast to the gradient type."""
    x = host_normal(n, std, seed, "grad", step, micro)
    x *= np.float32(scale)
    return host_cast(x, dtype)


WIDE_KINDS = ("mixed", "tiny", "subnormal", "max", "sparse_tiny")


def host_wide_range(n: int, seed: int, kind: str) -> np.ndarray:
    """float32 gradients whose magnitudes span the binary32 range, for the
    norm's range tests (cast to bfloat16 or kept as binary32):
      mixed       N(0, 1e-3^2), with 1 element in 1000 replaced by
                  +-U(1, 2) * 1e20 and 1 in 20 by +-U(1, 2) * 1e-30;
      tiny        N(0, 1) * 1e-25 everywhere;
      subnormal   N(0, 1) * 1e-40 everywhere (below binary32's normal range);
      max         +-U(0.5, 1) * 3.3e38 everywhere;
      sparse_tiny zero except 1 element in 100, +-U(1, 2) * 1e-30."""
    rng = np.random.default_rng(stream_seed(seed, "misc", n, WIDE_KINDS.index(kind)))
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    if kind == "mixed":
        x = rng.standard_normal(n) * GRAD_STD
        u = rng.random(n)
        x = np.where(u < 1e-3, sign * rng.uniform(1.0, 2.0, n) * 1e20, x)
        x = np.where((u >= 1e-3) & (u < 0.051), sign * rng.uniform(1.0, 2.0, n) * 1e-30, x)
    elif kind == "tiny":
        x = rng.standard_normal(n) * 1e-25
    elif kind == "subnormal":
        x = rng.standard_normal(n) * 1e-40
    elif kind == "max":
        x = sign * rng.uniform(0.5, 1.0, n) * 3.3e38
    elif kind == "sparse_tiny":
        x = np.where(rng.random(n) < 0.01, sign * rng.uniform(1.0, 2.0, n) * 1e-30, 0.0)
    else:
        raise ValueError(kind)
    return x.astype(np.float32)


def host_master(n: int, seed: int, std: float = MASTER_STD) -> np.ndarray:
    return host_normal(n, std, seed, "master")


def inf_index(n: int, seed: int, step: int) -> int:
    rng = np.random.default_rng(stream_seed(seed, "inf", step))
    return int(rng.integers(0, n))


def sample_indices(n: int, count: int, seed: int, edge: int = 4096) -> np.ndarray:
    """Sorted unique indices: the first and last ``edge`` elements plus
    ``count`` uniform draws."""
    rng = np.random.default_rng(stream_seed(seed, "sample", n))
    parts = [np.arange(min(edge, n)), np.arange(max(0, n - edge), n)]
    if n > 0:
        parts.append(rng.integers(0, n, size=count))
    return np.unique(np.concatenate(parts)).astype(np.int64)


# -- device-side draws (torch), for sizes the host would take long to draw


def _torch_dtype(dtype: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def device_normal(n: int, std: float, seed: int, stream: str, *keys: int, device="cuda",
                  chunk: int = 1 << 28):
    """n draws of N(0, std^2) as a float32 torch tensor on ``device``, from
    torch's generator seeded per stream (drawn in chunks of 2^28)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(stream_seed(seed, stream, *keys))
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e].normal_(0.0, 1.0, generator=gen)
    out.mul_(std)
    return out


def device_grad_into(out, seed: int, step: int, scale: float, micro: int = 0,
                     std: float = GRAD_STD, chunk: int = 1 << 28):
    """Fills ``out`` (a 1-D fp16/bf16/fp32 torch tensor) with the step's
    stored gradient N(0, std^2) * scale, drawn in float32 chunk by chunk."""
    import torch
    gen = torch.Generator(device=out.device)
    gen.manual_seed(stream_seed(seed, "grad", step, micro))
    n = out.numel()
    tmp = torch.empty(min(n, chunk), dtype=torch.float32, device=out.device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        t = tmp[: e - s]
        t.normal_(0.0, 1.0, generator=gen)
        t.mul_(std * scale)
        out[s:e].copy_(t)
    return out


def device_master_into(out, seed: int, std: float = MASTER_STD, chunk: int = 1 << 28):
    import torch
    gen = torch.Generator(device=out.device)
    gen.manual_seed(stream_seed(seed, "master"))
    n = out.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e].normal_(0.0, 1.0, generator=gen)
        out[s:e].mul_(std)
    return out
