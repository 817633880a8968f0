"""The GPU parity harness's derived bounds, checked on the CPU.

When the GPU's binary32 clip coefficient rounds one ulp away from the
oracle's (their norms are summed in different orders), the element
comparison uses per-element bounds carried through the update's arithmetic
(gpu_common.oracle_step / _propagate).  Here a stand-in for the GPU is the
oracle itself with its first step's clip coefficient moved by one ulp: every
element of its state must lie within the derived bounds over several steps,
many of them beyond the plain 1e-6 relative bar (the update cancelling the
master), while a planted error of a few millionths in one element is caught."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

gc = pytest.importorskip("gpu_common")


def _run(n, steps, bump, plant=None):
    hp = oracle.HParams(max_norm=0.05)
    scale = 1024.0
    p0 = zs.host_master(n, 5)
    ref = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    gpu = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    sc_ref, sc_gpu = oracle.Scaler(loss_scale=scale), oracle.Scaler(loss_scale=scale)
    beyond_bar = 0
    for k in range(steps):
        g = zs.host_grad(n, 5, k, scale, "f16")
        # the stand-in: the oracle's own step, its clip coefficient moved by
        # `bump` ulps at the first step
        sumsq, bad = oracle.norm_overflow([g], "f16", scale)
        st_g = oracle.decide(hp, sc_gpu, sumsq, bad)
        if k == 0 and bump:
            st_g = oracle.with_clip(st_g, float(np.nextafter(np.float32(st_g.scalars["clip"]),
                                                             np.float32(np.inf * bump))))
        oracle.adam_apply(g, "f16", gpu[0], gpu[1], gpu[2], gpu[3], "f16", st_g)
        if plant is not None and k == plant[0]:
            gpu[0][plant[1]] *= np.float32(1 + plant[2])
        state = {"last_skipped": 0, "step": sc_gpu.step, "loss_scale": sc_gpu.loss_scale,
                 "good_steps": sc_gpu.good_steps, "last_norm": st_g.norm,
                 "last_clip": st_g.scalars["clip"]}
        st = gc.oracle_step([g], "f16", [ref[0]], [ref[1]], [ref[2]], [ref[3]], "f16", hp, sc_ref, state)
        assert st.exact == (bump == 0)
        for name, i in (("p", 0), ("m", 1), ("v", 2)):
            gc.assert_f32(gpu[i], ref[i], f"{name} step {k}", st.exact, gc.bound_of(st, name, 0))
            b = gc.bound_of(st, name, 0)
            if b is not None:
                beyond_bar += gc._tight(gpu[i], ref[i], b)
        gc.assert_lp(gpu[3], ref[0], "f16", f"p_lp step {k}", st.exact, gc.bound_of(st, "p", 0))
    return beyond_bar


@pytest.fixture(autouse=True)
def _keep_the_session_record():
    """These stand-in runs are not GPU comparisons: the session's parity
    record is left as it was."""
    saved = (gc.Parity.steps, gc.Parity.clip_differs, gc.Parity.tight, gc.Parity.bounded)
    yield
    gc.Parity.steps, gc.Parity.clip_differs, gc.Parity.tight, gc.Parity.bounded = saved


@pytest.mark.parametrize("bump", [1, -1])
def test_one_ulp_clip_difference_stays_within_the_derived_bounds(bump):
    # elements whose update cancels the master go beyond the plain bar but
    # stay within the bound (the case the bound exists for)
    assert _run(200_003, 4, bump) > 0


def test_same_clip_is_held_bit_for_bit():
    assert _run(20_001, 3, 0) == 0


@pytest.mark.parametrize("rel", [1e-5, -3e-6])
def test_a_planted_error_is_caught(rel):
    """One master element off by a few millionths (beyond the bar, far
    beyond what a one-ulp clip difference explains) after the step whose
    clip coefficient differed."""
    with pytest.raises(AssertionError, match="master|p step"):
        _run(20_001, 3, 1, plant=(1, 1234, rel))
