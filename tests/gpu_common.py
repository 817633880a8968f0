"""Shared helpers of the GPU parity tests: run a shard through the C ABI and
the oracle side by side and compare.

The bar (element by element):
  * fp32 master, momentum, variance: within 1e-6 relative + 1e-12 absolute of
    the oracle, and in fact bit-identical whenever both sides use the same
    binary32 step scalars (the kernels evaluate the oracle's expression with
    the same IEEE operations in the same order);
  * fp16/bf16 parameters: within 1 ulp of the oracle master rounded to
    nearest even (and bit-identical);
  * skip decision, step count, loss scale: identical;
  * global norm: within 1e-6 relative of the oracle's binary64 sum.
The norm's summation order differs between the two sides, so the binary32
clip coefficient derived from it can in rare cases round the other way; the
comparison then checks the norms agree and follows the GPU's coefficient for
the element update (``oracle.with_clip``)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import zero_partitioned_mixed_layout_gb300 as zp

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
REL, ABS = 1e-6, 1e-12
NORM_REL = 1e-6


def to_dev(a: np.ndarray, dtype: str, dev="cuda"):
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def to_host(t) -> np.ndarray:
    """Raw host copy: float32 as float32, 16-bit types as uint16 bit patterns."""
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def hp_pair(**kw):
    return oracle.HParams(**kw), zp.HParams(**kw)


def assert_f32(gpu: np.ndarray, ref: np.ndarray, what: str, exact: bool = True):
    g64, r64 = gpu.astype(np.float64), ref.astype(np.float64)
    bad = ~(np.abs(g64 - r64) <= REL * np.abs(r64) + ABS)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside 1e-6 rel + 1e-12 abs; "
                             f"first at {i}: gpu {gpu[i]!r} oracle {ref[i]!r}")
    if exact:
        diff = gpu.view(np.uint32) != ref.view(np.uint32)
        if diff.any():
            i = int(np.flatnonzero(diff)[0])
            raise AssertionError(f"{what}: {int(diff.sum())} elements not bit-identical; first at "
                                 f"{i}: gpu {gpu[i]!r} oracle {ref[i]!r}")


def assert_lp(gpu_bits: np.ndarray, ref_master: np.ndarray, pdtype: str, what: str):
    ref_bits = oracle.to_lp(ref_master, pdtype)
    # within one ulp: same sign and adjacent patterns (patterns are monotone per sign)
    d = np.abs(gpu_bits.astype(np.int64) - ref_bits.astype(np.int64))
    same_sign = (gpu_bits >> 15) == (ref_bits >> 15)
    ok = (d <= 1) & same_sign | ((gpu_bits & 0x7FFF) == 0) & ((ref_bits & 0x7FFF) == 0)
    assert ok.all(), f"{what}: {int((~ok).sum())} low-precision params beyond 1 ulp"
    assert np.array_equal(gpu_bits, ref_bits), f"{what}: low-precision params not bit-identical"


class Mismatch:
    clip_followed = 0


def oracle_step(grads, gdtype, p, m, v, plp, pdtype, hp, sc, gpu_state, sampled_idx=None):
    """The oracle's step on host arrays, checked against the GPU's decision."""
    sumsq, bad = oracle.norm_overflow(grads, gdtype, sc.loss_scale)
    st = oracle.decide(hp, sc, sumsq, bad)
    assert bool(gpu_state["last_skipped"]) == st.skip, "skip decision differs"
    assert gpu_state["step"] == sc.step, "step count differs"
    assert gpu_state["loss_scale"] == sc.loss_scale, "loss scale differs"
    assert gpu_state["good_steps"] == sc.good_steps
    if not st.skip:
        assert abs(gpu_state["last_norm"] - st.norm) <= NORM_REL * st.norm, (
            f"norm differs: gpu {gpu_state['last_norm']!r} oracle {st.norm!r}")
        gclip = np.float32(gpu_state["last_clip"])
        if gclip != np.float32(st.scalars["clip"]):
            Mismatch.clip_followed += 1
            st = oracle.with_clip(st, float(gclip))
    if sampled_idx is None:
        for i, g in enumerate(grads):
            oracle.adam_apply(g, gdtype, p[i], m[i], v[i], plp[i], pdtype, st)
    else:
        oracle.adam_apply_sampled(grads[0], gdtype, sampled_idx, p[0], m[0], v[0], plp[0],
                                  pdtype, st)
    return st
