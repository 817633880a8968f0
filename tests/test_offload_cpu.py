"""The ZeRO-Offload host step (zero_offload_decide / zero_offload_apply) on
the CPU against the oracle: the same decisions and the same bits, on every
element type, with 1 to 8 host threads, whole or chunk by chunk."""
import numpy as np
import pytest

import oracle
import zero_synth as zs


@pytest.fixture(scope="module")
def zp():
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def host_state(zp, scale, step=0, good=0, sumsq=0.0, found_inf=0.0):
    st = np.frombuffer(bytearray(zp.zero_state_init(scale)), dtype=np.uint8).copy()
    f = st.view(np.float64)
    f[0], f[1] = sumsq, found_inf
    i = st.view(np.int64)
    i[3], i[4] = step, good
    return st


CASES = [dict(sumsq=2.5e-3, found_inf=0.0, scale=1024.0, step=0, good=0, hp={}),
         dict(sumsq=4.0, found_inf=0.0, scale=65536.0, step=7, good=999, hp=dict(max_norm=1.0)),
         dict(sumsq=1e-9, found_inf=0.0, scale=1.0, step=4999, good=3, hp=dict(max_norm=1.0)),
         dict(sumsq=np.inf, found_inf=1.0, scale=2.0, step=3, good=5, hp=dict(max_norm=1.0)),
         dict(sumsq=0.3, found_inf=2.0, scale=1.0, step=0, good=0, hp={})]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decide_matches_oracle(zp, case):
    c = CASES[case]
    st = host_state(zp, c["scale"], c["step"], c["good"], c["sumsq"], c["found_inf"])
    sc = zp.zero_offload_decide(st, zp.HParams(**c["hp"]))
    osc = oracle.Scaler(loss_scale=c["scale"], step=c["step"], good_steps=c["good"])
    ost = oracle.decide(oracle.HParams(**c["hp"]), osc, c["sumsq"], int(c["found_inf"] > 0))
    got = zp.parse_state(st)
    assert bool(sc.skip) == ost.skip
    assert got["loss_scale"] == osc.loss_scale and got["step"] == osc.step
    assert got["good_steps"] == osc.good_steps and got["sumsq"] == 0.0 and got["found_inf"] == 0.0
    if not ost.skip:
        names = {"inv_scale": "inv_scale", "clip": "clip", "beta1": "beta1",
                 "one_minus_beta1": "one_minus_beta1", "beta2": "beta2",
                 "one_minus_beta2": "one_minus_beta2", "eps": "eps", "step_size": "step_size",
                 "inv_sqrt_bc2": "inv_sqrt_bc2", "lr_wd": "lr_wd"}
        for ours, theirs in names.items():
            assert np.float32(getattr(sc, ours)) == np.float32(ost.scalars[theirs]), ours


@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "bf16"),
                                           ("f32", "f16")])
@pytest.mark.parametrize("n", [1, 7, 65536, 65537, 300_001])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_apply_matches_oracle(zp, gdtype, pdtype, n, threads):
    scale = 1024.0 if gdtype == "f16" else 1.0
    hp = dict(max_norm=0.05)
    rng_state = host_state(zp, scale, step=2)
    p0 = zs.host_master(n, n)
    m0 = zs.host_normal(n, 1e-4, n, "misc", 1)
    v0 = np.abs(zs.host_normal(n, 1e-7, n, "misc", 2))
    g = zs.host_grad(n, n, 0, scale, gdtype)
    sumsq, bad = oracle.norm_overflow([g], gdtype, scale)
    f = rng_state.view(np.float64)
    f[0], f[1] = sumsq, float(bad)
    sc = zp.zero_offload_decide(rng_state, zp.HParams(**hp))
    p, m, v = p0.copy(), m0.copy(), v0.copy()
    lp = np.zeros(n, np.uint16)
    gview = g.view(np.uint16) if gdtype == "f16" else g
    zp.zero_offload_apply(gview, p, m, v, lp, sc, gdtype=gdtype, pdtype=pdtype, n_threads=threads)
    ost = oracle.decide(oracle.HParams(**hp), oracle.Scaler(loss_scale=scale, step=2), sumsq, bad)
    rp, rm, rv = p0.copy(), m0.copy(), v0.copy()
    rlp = np.zeros(n, np.uint16)
    oracle.adam_apply(g, gdtype, rp, rm, rv, rlp, pdtype, ost)
    for a, b in ((p, rp), (m, rm), (v, rv), (lp, rlp)):
        assert a.tobytes() == b.tobytes()


def test_chunked_apply_equals_whole_and_skip(zp):
    n = 1_000_003
    g = zs.host_grad(n, 9, 0, 1024.0, "f16").view(np.uint16)
    st = host_state(zp, 1024.0, sumsq=0.7)
    sc = zp.zero_offload_decide(st, zp.HParams())
    p0 = zs.host_master(n, 9)
    a = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    b = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    zp.zero_offload_apply(g, *a, sc, gdtype="f16", pdtype="f16")
    cuts = [0, 5, 70_000, 70_001, 500_000, n]
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        zp.zero_offload_apply(g[lo:hi], *[x[lo:hi] for x in b], sc, gdtype="f16", pdtype="f16",
                              n_threads=4)
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()
    # a skipped step touches nothing
    st = host_state(zp, 1024.0, found_inf=1.0)
    sc = zp.zero_offload_decide(st, zp.HParams())
    before = [x.copy() for x in a]
    zp.zero_offload_apply(g, *a, sc, gdtype="f16", pdtype="f16")
    assert sc.skip == 1 and all(x.tobytes() == y.tobytes() for x, y in zip(a, before))
    assert zp.parse_state(st)["loss_scale"] == 512.0


def test_offload_steps_follow_oracle(zp):
    """Three steps (the second overflows) of the host step against the
    oracle's full step, gradient norm formed with the oracle's pass 1."""
    n = 200_003
    scale = 1024.0
    st = host_state(zp, scale)
    p, m, v, lp = zs.host_master(n, 4), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    rp, rm, rv, rlp = p.copy(), m.copy(), v.copy(), lp.copy()
    sc_o = oracle.Scaler(loss_scale=scale)
    hp = dict(max_norm=0.5)
    for k in range(3):
        cur = zp.parse_state(st)["loss_scale"]
        g = zs.host_grad(n, 4, k, cur, "f16")
        if k == 1:
            g[17] = np.inf
        sumsq, bad = oracle.norm_overflow([g], "f16", cur)
        f = st.view(np.float64)
        f[0], f[1] = sumsq, float(bad)
        sc = zp.zero_offload_decide(st, zp.HParams(**hp))
        zp.zero_offload_apply(g.view(np.uint16), p, m, v, lp, sc, gdtype="f16", pdtype="f16")
        oracle.adam_step([g], "f16", [rp], [rm], [rv], [rlp], "f16", oracle.HParams(**hp), sc_o)
        assert zp.parse_state(st)["step"] == sc_o.step
        assert zp.parse_state(st)["loss_scale"] == sc_o.loss_scale
    for a, b in ((p, rp), (m, rm), (v, rv), (lp, rlp)):
        assert a.tobytes() == b.tobytes()


def test_copy_and_errors(zp):
    src = np.random.default_rng(0).integers(0, 255, 5_000_003).astype(np.uint8)
    dst = np.zeros_like(src)
    zp.zero_offload_copy(dst, src, n_threads=5)
    assert np.array_equal(dst, src)
    with pytest.raises(zp.ZeroError):
        zp.zero_offload_apply(np.zeros(4, np.float16), np.zeros(4, np.float32), np.zeros(4, np.float32),
                              np.zeros(4, np.float32), None, zp.OffloadScalars(), n_threads=-1)


def test_every_f16_gradient_value_converts_exactly(zp):
    """All 63,488 finite binary16 values (and +-inf) through the host update
    with beta1 = 0 and no loss scale: the new momentum is the gradient's
    binary32 value, which must equal numpy's exact conversion."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7C00) != 0x7C00
    infs = (bits & 0x7FFF) == 0x7C00
    keep = bits[finite | infs]
    g = keep.view(np.float16)
    n = g.size
    st = host_state(zp, 1.0)
    sc = zp.zero_offload_decide(st, zp.HParams(beta1=0.0))
    p = np.zeros(n, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    zp.zero_offload_apply(np.ascontiguousarray(g), p, m, v, None, sc, n_threads=2)
    # m' = 0*0 + 1*g: -0 comes out as +0 (0 + -0 = +0), every other value as is
    want = np.float32(0.0) + g.astype(np.float32)
    assert m.tobytes() == want.tobytes()


def test_decide_refuses_a_scale_floor_that_is_not_a_power_of_two(zp):
    """Halving down to a floor that is not a power of two would leave a loss
    scale whose reciprocal is inexact: such a floor is refused."""
    st = host_state(zp, 1024.0, found_inf=1.0)
    with pytest.raises(zp.ZeroError) as e:
        zp.zero_offload_decide(st, zp.HParams(min_scale=3.0))
    assert e.value.code == -1
    sc = zp.zero_offload_decide(st, zp.HParams(min_scale=4.0))
    assert sc is not None
