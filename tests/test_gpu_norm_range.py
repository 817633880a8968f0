"""Pass 1 over bfloat16 and binary32 gradients whose magnitudes span the
binary32 range, against the oracle's binary64 sum of squares.

Binary16 values square into binary32's normal range whatever they are;
bfloat16 and binary32 values do not: a finite value above 2^64 squares to
inf in binary32, one below 2^-63 loses digits or vanishes.  The kernels sum
squares in binary32 per 8 elements and fall back to binary64 for a vector
whose binary32 sum is out of range.  These tests feed that range -- values
near 1e20 among ordinary ones, every value tiny, subnormal or near the
binary32 maximum, a sparse scatter of tiny values -- through each kernel that
squares (pass 1 on a flat shard and on a list, the fused accumulation, the
stage-2 reduction) and hold the norm to the oracle's within 1e-6; the whole
step with clipping on is then compared element by element (bit-identical
while the two sides' clip coefficients agree)."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import (bound_of, NORM_REL, assert_f32, assert_lp, assert_lp_copy, hp_pair, oracle_step,  # noqa: E402
                        to_dev, to_host)


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def norm_of(zp, state):
    st = zp.parse_state(state)
    return st["sumsq"], st["found_inf"]


def check_norm(gpu_sumsq, ora_sumsq, what):
    assert np.isfinite(gpu_sumsq), f"{what}: the GPU's sum of squares is {gpu_sumsq!r}"
    g, o = np.sqrt(gpu_sumsq), np.sqrt(ora_sumsq)
    assert abs(g - o) <= NORM_REL * o, f"{what}: norm gpu {g!r} oracle {o!r}"


SIZES = {"flat": [100_003], "list": [5, 70_001, 3, 33, 4096]}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kind", zs.WIDE_KINDS)
@pytest.mark.parametrize("layout", ["flat", "list"])
def test_pass1_norm_over_the_binary32_range(zp, dtype, kind, layout):
    host = [zs.host_cast(zs.host_wide_range(n, 60 + i, kind), dtype) for i, n in enumerate(SIZES[layout])]
    dev = [to_dev(a, dtype) for a in host]
    state, ws = zp.new_state(1.0), zp.new_workspace(len(dev), sum(SIZES[layout]))
    zp.zero_grad_norm_overflow(dev if layout == "list" else dev[0], state, ws)
    sumsq, found = norm_of(zp, state)
    ora_sumsq, ora_bad = oracle.norm_overflow(host, dtype, 1.0)
    assert found == 0.0 and ora_bad == 0
    assert ora_sumsq > 0.0
    check_norm(sumsq, ora_sumsq, f"{kind} {dtype} {layout}")


@pytest.mark.parametrize("gdtype,pdtype", [("bf16", "bf16"), ("f32", "f16")])
@pytest.mark.parametrize("whole", [True, False], ids=["zero_step", "two_calls"])
def test_step_with_huge_gradients_matches_oracle(zp, gdtype, pdtype, whole):
    """Three steps with clipping at 1.0 on gradients that hold values near
    1e20 (and near 1e-30): the norm stays finite, so the clip coefficient is
    the oracle's and every element follows it."""
    n = 100_003
    ohp, ghp = hp_pair(max_norm=1.0)
    p0 = zs.host_master(n, 61)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm, dv = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    dlp = torch.zeros(n, dtype={"bf16": torch.bfloat16, "f16": torch.float16}[pdtype], device="cuda")
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    p, m, v, plp = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=1.0)
    for k in range(3):
        g = zs.host_cast(zs.host_wide_range(n, 62 + k, "mixed"), gdtype)
        dg = to_dev(g, gdtype)
        if whole:
            zp.zero_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        else:
            zp.zero_grad_norm_overflow(dg, state, ws)
            zp.zero_adam_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step([g], gdtype, [p], [m], [v], [plp], pdtype, ohp, sc, gst)
        assert not st.skip and st.norm > 1e20 and st.scalars["clip"] < 1e-19
        assert_f32(to_host(dp), p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(to_host(dm), m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(to_host(dv), v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp_copy(to_host(dlp), plp, f"p_lp step {k}", st.exact)
        assert_lp(to_host(dlp), p, pdtype, f"p_lp step {k}", st.exact, bound_of(st, "p", 0))


@pytest.mark.parametrize("kind", ["mixed", "tiny", "sparse_tiny"])
def test_fused_accumulation_norm_over_the_range(zp, kind):
    """Four bfloat16 micro-batches summed into binary32 with pass 1 fused:
    the sums bit for bit, the norm of the stored sums within 1e-6."""
    n, micro = 100_003, 4
    bufs = [zs.host_cast(zs.host_wide_range(n, 70 + j, kind), "bf16") for j in range(micro)]
    acc = np.zeros(n, np.float32)
    oracle.accumulate(acc, bufs, "bf16", True)
    dacc = torch.empty(n, dtype=torch.float32, device="cuda")
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    zp.zero_accumulate_grads_norm(dacc, [to_dev(b, "bf16") for b in bufs], state, ws, True)
    assert to_host(dacc).tobytes() == acc.tobytes()
    sumsq, found = norm_of(zp, state)
    ora_sumsq, ora_bad = oracle.norm_overflow([acc], "f32", 1.0)
    assert found == 0.0 and ora_bad == 0
    check_norm(sumsq, ora_sumsq, f"accumulation {kind}")


@pytest.mark.parametrize("kind", ["mixed", "tiny", "sparse_tiny"])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_stage2_reduction_norm_over_the_range(zp, kind, out_dtype):
    """The stage-2 mean of four bfloat16 replicas: the stored mean bit for
    bit, the norm of the stored mean within 1e-6."""
    n, nr = 100_003, 4
    reps = [zs.host_cast(zs.host_wide_range(n, 80 + r, kind), "bf16") for r in range(nr)]
    mean = oracle.reduce_mean(reps, "bf16", out_dtype)
    out = torch.empty(n, dtype={"bf16": torch.bfloat16, "f32": torch.float32}[out_dtype], device="cuda")
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    zp.zero_reduce_grads([to_dev(r, "bf16") for r in reps], out, state, ws)
    assert to_host(out).tobytes() == mean.tobytes()
    sumsq, found = norm_of(zp, state)
    ora_sumsq, ora_bad = oracle.norm_overflow([mean], out_dtype, 1.0)
    assert found == 0.0 and ora_bad == 0
    check_norm(sumsq, ora_sumsq, f"stage-2 mean {kind} {out_dtype}")
