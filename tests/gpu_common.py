"""Shared helpers of the GPU parity tests: run a shard through the C ABI and
the oracle side by side and compare.

The oracle runs on its own: it takes its own decision (skip, loss scale, norm,
clip coefficient) from the seeded inputs, and nothing computed on the GPU is
fed into it.  The bar (element by element):
  * fp32 master, momentum, variance: within 1e-6 relative + 1e-12 absolute of
    the oracle;
  * fp16/bf16 parameters: within 1 ulp of the oracle master rounded to
    nearest even;
  * skip decision, step count, loss scale: identical;
  * global norm: within 1e-6 relative of the oracle's binary64 sum.
Beyond the bar, the element update must be bit-identical to the oracle's
whenever both sides applied the same binary32 clip coefficient at this step
and at every earlier step of the sequence: the kernels evaluate the oracle's
expression with the same IEEE operations in the same order.  The norm is
summed in another order on the two sides, so the binary32 clip coefficient
derived from it can round the other way (it did not in any run so far); from
such a step on the comparison is the tolerance above.  ``Parity`` counts the
steps compared and those whose coefficients differed; the count is printed
at the end of the session."""
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


U32 = 2.0 ** -24  # unit roundoff of binary32


def _tight(gpu, ref, bound):
    """Elements beyond the bar but within the derived bound (counted)."""
    d = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    return int(np.sum(d > REL * np.abs(ref.astype(np.float64)) + ABS))


def assert_f32(gpu: np.ndarray, ref: np.ndarray, what: str, exact: bool = True, bound=None):
    """Within 1e-6 relative + 1e-12 absolute, or within ``bound`` (a
    per-element absolute bound derived from a clip coefficient that rounded
    the other way, see ``oracle_step``) where that is larger; bit-identical
    when ``exact``."""
    g64, r64 = gpu.astype(np.float64), ref.astype(np.float64)
    allow = REL * np.abs(r64) + ABS
    if bound is not None:
        allow = np.maximum(allow, bound)
        Parity.tight += _tight(gpu, ref, bound)
        Parity.bounded += int(gpu.size)
    bad = ~(np.abs(g64 - r64) <= allow)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        extra = f" (derived bound {bound[i]!r})" if bound is not None else ""
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside 1e-6 rel + 1e-12 abs; "
                             f"first at {i}: gpu {gpu[i]!r} oracle {ref[i]!r}{extra}")
    if exact:
        diff = gpu.view(np.uint32) != ref.view(np.uint32)
        if diff.any():
            i = int(np.flatnonzero(diff)[0])
            raise AssertionError(f"{what}: {int(diff.sum())} elements not bit-identical; first at "
                                 f"{i}: gpu {gpu[i]!r} oracle {ref[i]!r}")


def within_one_ulp(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Per element: two binary16 / bfloat16 bit patterns are equal or
    adjacent values (patterns are monotone within a sign; the two zeros are
    one value)."""
    d = np.abs(a_bits.astype(np.int64) - b_bits.astype(np.int64))
    same_sign = (a_bits >> 15) == (b_bits >> 15)
    zeros = ((a_bits & 0x7FFF) == 0) & ((b_bits & 0x7FFF) == 0)
    return ((d <= 1) & same_sign) | zeros


def _lp_ok(gpu_bits, ref_bits, pdtype, ref_master, bound):
    """Within 1 ulp, or -- where a derived bound on the master applies -- the
    GPU's low-precision value within that bound plus one of its own ulps of
    the oracle master."""
    ok = within_one_ulp(gpu_bits, ref_bits)
    if bound is not None and ref_master is not None:
        gv = oracle.from_lp(gpu_bits, pdtype).astype(np.float64)
        ulp = np.abs(gv) * (2.0 ** -10 if pdtype == "f16" else 2.0 ** -7) + 2.0 ** -24
        ok |= np.abs(gv - ref_master.astype(np.float64)) <= bound + ulp
    return ok


def assert_lp(gpu_bits: np.ndarray, ref_master: np.ndarray, pdtype: str, what: str, exact: bool = True,
              bound=None):
    """Within 1 ulp of the oracle master rounded to nearest even (or within
    the master's derived bound, see assert_f32); bit-identical when
    ``exact``."""
    ref_bits = oracle.to_lp(ref_master, pdtype)
    ok = _lp_ok(gpu_bits, ref_bits, pdtype, ref_master, bound)
    assert ok.all(), f"{what}: {int((~ok).sum())} low-precision params beyond 1 ulp"
    if exact:
        assert np.array_equal(gpu_bits, ref_bits), f"{what}: low-precision params not bit-identical"


def assert_lp_copy(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str, exact: bool = True):
    """The low-precision copy against the oracle's own copy (which a skipped
    step leaves alone): bit-identical when ``exact``, else not compared here
    (assert_lp holds it to the oracle master)."""
    if exact:
        assert np.array_equal(gpu_bits, ref_bits), f"{what}: low-precision params not bit-identical"


class Parity:
    """Steps compared in this session, those whose binary32 clip coefficient
    differed between the GPU and the oracle, and the elements that needed
    the derived bound (beyond 1e-6 relative + 1e-12 absolute)."""
    steps = 0
    clip_differs = 0
    tight = 0
    bounded = 0  # elements compared under a derived bound


class Bounds:
    """Per-element bounds on |GPU - oracle| of one sequence's arrays (lists
    of float64 arrays, one per array of the step), carried from step to step
    once the two sides' clip coefficients have differed."""

    def __init__(self, n_arrays):
        self.p = [None] * n_arrays
        self.m = [None] * n_arrays
        self.v = [None] * n_arrays


def _grad_magnitude(g, gdtype, idx, inv_scale):
    """|float(g_lp) * (1/S)| in binary64 (exact: a power-of-two scale)."""
    a = np.ascontiguousarray(g if idx is None else g[idx])
    f = a.astype(np.float64) if gdtype == "f32" else oracle.from_lp(a, gdtype).astype(np.float64)
    return np.abs(f) * float(inv_scale)


def _propagate(sc_, gu, p0, m0, v0, p1, m1, v1, Dp, Dm, Dv, dclip):
    """Bounds on |GPU - oracle| of p, m, v after one applied step, from the
    bounds entering it and the bound dclip on the difference of the two
    sides' binary32 clip coefficients.  Each operation of the element update
    (binary32, in the order the kernels and the oracle share) is followed by
    the exact sensitivity of its result to its inputs (triangle
    inequalities) plus, where any input differs, a rounding allowance: each
    rounding moves its result by at most one unit roundoff u of it, on each
    side, and the allowance is 2.5u (2u and slack) times the magnitude that
    rounding contributes to the result.  Where no input differs the two
    sides compute the same bits and the bound is 0."""
    b1, omb1 = float(sc_["beta1"]), float(sc_["one_minus_beta1"])
    b2, omb2 = float(sc_["beta2"]), float(sc_["one_minus_beta2"])
    isb2, eps = float(sc_["inv_sqrt_bc2"]), float(sc_["eps"])
    ss, lrwd, c = float(sc_["step_size"]), float(sc_["lr_wd"]), float(sc_["clip"])
    R = 2.5 * U32
    f = lambda a: np.abs(np.asarray(a, np.float64))  # noqa: E731
    p0, m0, v0, p1, m1, v1 = f(p0), f(m0), f(v0), f(p1), f(m1), f(v1)
    # g = (g_lp * (1/S)) * clip: the first product is exact, the second
    # rounds; with different clip coefficients the two sides' g differ
    g = gu * c
    Dg = gu * dclip + (R * g if dclip > 0 else 0.0)
    r = ((Dm > 0) | (Dv > 0) | (Dp > 0) | (Dg > 0)).astype(np.float64)
    # m' = b1*m + omb1*g: two products and a sum
    Dm1 = b1 * Dm + omb1 * Dg + r * R * (b1 * m0 + omb1 * g + m1)
    # v' = b2*v + omb2*(g*g): three products and a sum
    Dv1 = b2 * Dv + omb2 * (2 * g * Dg + Dg * Dg) + r * R * (b2 * v0 + 2 * omb2 * g * g + v1)
    # d = sqrt(v')*isb2 + eps: |sqrt(a) - sqrt(b)| <= |a - b| / sqrt(a) and
    # <= sqrt(|a - b|); the square root, product and sum each round
    sq = np.sqrt(v1)
    with np.errstate(divide="ignore", invalid="ignore"):
        dsq = np.minimum(np.sqrt(Dv1), np.where(sq > 0, Dv1 / sq, np.inf))
    d = sq * isb2 + eps
    Dd = isb2 * dsq + r * R * (2 * sq * isb2 + d)
    # u = m'/d
    u = m1 / d
    with np.errstate(divide="ignore", invalid="ignore"):
        Du = np.where(d > Dd, (Dm1 + u * Dd) / (d - Dd), np.inf) + r * R * u
    # p' = p - (step_size*u + lrwd*p): dp'/dp = 1 - lrwd; two products, a
    # sum and a difference
    Dp1 = Dp + ss * Du + r * R * (2 * (ss * u + lrwd * p0) + p1)
    return Dp1, Dm1, Dv1


def oracle_step(grads, gdtype, p, m, v, plp, pdtype, hp, sc, gpu_state, sampled_idx=None):
    """The oracle's step on host arrays, with its own decision, checked
    against the GPU's decision (skip, step count, loss scale, norm).  Returns
    the oracle's Step.  Its ``exact`` attribute says whether the elements may
    be held to bit identity: the two sides applied the same binary32 clip
    coefficient at this step and at every earlier step of this sequence.
    Once they have not, ``bounds`` holds per-element bounds on |GPU - oracle|
    for p, m and v (see _propagate), sized by the difference of the two
    binary32 coefficients -- itself held to what the norm tolerance allows:
    max_norm / (norm + 1e-6) of two norms within 1e-6 of each other differ by
    at most 1e-6 relative plus one rounding on each side.  ``sc`` carries the
    record from step to step.  Nothing the GPU computed enters the oracle's
    arithmetic: the GPU's coefficient only sizes the comparison's bound."""
    sumsq, bad = oracle.norm_overflow(grads, gdtype, sc.loss_scale)
    inv_scale = np.float32(1.0 / sc.loss_scale)
    st = oracle.decide(hp, sc, sumsq, bad)
    assert bool(gpu_state["last_skipped"]) == st.skip, "skip decision differs"
    assert gpu_state["step"] == sc.step, "step count differs"
    assert gpu_state["loss_scale"] == sc.loss_scale, "loss scale differs"
    assert gpu_state["good_steps"] == sc.good_steps
    n_arrays = len(grads) if sampled_idx is None else 1
    bounds = getattr(sc, "gpu_bounds", None)
    dclip = 0.0
    if not st.skip:
        assert abs(gpu_state["last_norm"] - st.norm) <= NORM_REL * st.norm, (
            f"norm differs: gpu {gpu_state['last_norm']!r} oracle {st.norm!r}")
        Parity.steps += 1
        c_gpu, c_ora = np.float32(gpu_state["last_clip"]), np.float32(st.scalars["clip"])
        if c_gpu != c_ora:
            Parity.clip_differs += 1
            dclip = abs(float(c_gpu) - float(c_ora))
            # what two norms within the tolerance allow: max_norm/(norm + 1e-6)
            # moves by at most NORM_REL relative, plus a rounding on each side
            assert dclip <= (NORM_REL + 4 * U32) * float(c_ora), (
                f"clip coefficient differs beyond the norm tolerance: gpu {c_gpu!r} oracle {c_ora!r}")
            if bounds is None:
                bounds = Bounds(n_arrays)
    keep = [] if bounds is None or st.skip else [(p[i].copy(), m[i].copy(), v[i].copy()) for i in range(n_arrays)]
    if sampled_idx is None:
        for i, g in enumerate(grads):
            oracle.adam_apply(g, gdtype, p[i], m[i], v[i], plp[i], pdtype, st)
    else:
        oracle.adam_apply_sampled(grads[0], gdtype, sampled_idx, p[0], m[0], v[0], plp[0],
                                  pdtype, st)
    for i, (p0, m0, v0) in enumerate(keep):
        z = np.zeros(p0.size)
        gu = _grad_magnitude(grads[i] if sampled_idx is None else grads[0], gdtype, sampled_idx, inv_scale)
        bounds.p[i], bounds.m[i], bounds.v[i] = _propagate(
            st.scalars, gu, p0, m0, v0, p[i], m[i], v[i],
            z if bounds.p[i] is None else bounds.p[i], z if bounds.m[i] is None else bounds.m[i],
            z if bounds.v[i] is None else bounds.v[i], dclip)
    sc.gpu_bounds = bounds
    st.exact = bounds is None
    st.bounds = bounds
    return st


def bound_of(st, name: str, i: int = 0):
    """The derived bound of array `name` ("p", "m" or "v") number i of a step
    returned by oracle_step, or None while the sequence is exact."""
    b = getattr(st, "bounds", None)
    return None if b is None else getattr(b, name)[i]
