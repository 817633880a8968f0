"""Pins for the oracle: each test checks it against something other than
itself -- closed forms of Adam, the textbook update in binary64 within a
derived rounding bound, torch's AdamW, exact sums, numpy/torch casts, and the
numbers the ZeRO pages print.  CPU only."""
import math

import numpy as np
import pytest

import oracle
import zero_synth as zs

U32 = 2.0 ** -24  # unit roundoff of binary32


def f16(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def step_once(g_lp, gdtype, p, m, v, hp, sc, pdtype="f16"):
    plp = np.zeros(p.size, np.uint16)
    st = oracle.adam_step([g_lp], gdtype, [p], [m], [v], [plp], pdtype, hp, sc)
    return st, plp


# ---------------------------------------------------------------- casts

def test_f16_cast_matches_numpy():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 5, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -26, np.inf, -np.inf], np.float32),
        # exact ties between neighbouring binary16 values
        (np.arange(1, 2000, dtype=np.float32) * 2 + 1) * np.float32(2.0 ** -11) + np.float32(1.0),
    ]).astype(np.float32)
    ours = oracle.to_lp(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.from_lp(ours, "f16")
    assert np.array_equal(back, ref.view(np.float16).astype(np.float32))


def test_bf16_cast_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 3.389e38, 3.4e38, -3.4e38, 1e-40, np.inf, -np.inf], np.float32),
        # ties: binary32 patterns whose low 16 bits are exactly 0x8000
        (np.arange(0, 4000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
    ]).astype(np.float32)
    ours = oracle.to_lp(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(oracle.from_lp(ours, "bf16"),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("eps", [0.0, 1e-8])
def test_step1_closed_form(eps):
    """t = 1 from m = v = 0: m_hat = g and v_hat = g^2, so
    p1 = p - lr * (g / (|g| + eps) + wd * p); with eps = 0 the Adam part is
    exactly -lr * sign(g)."""
    n = 50000
    rng = np.random.default_rng(3)
    scale = 1024.0
    g_true = rng.standard_normal(n).astype(np.float32) * np.float32(1e-3)
    g_lp = f16(g_true * scale)
    keep = g_lp != 0
    g_lp = np.ascontiguousarray(g_lp[keep])
    n = g_lp.size
    p0 = rng.standard_normal(n).astype(np.float32) * np.float32(0.02)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = oracle.HParams(eps=eps)
    st, _ = step_once(g_lp, "f16", p, m, v, hp, oracle.Scaler(loss_scale=scale))
    assert not st.skip
    g = g_lp.astype(np.float64) / scale
    expect = p0.astype(np.float64) - hp.lr * (g / (np.abs(g) + eps) + hp.weight_decay * p0)
    err = np.abs(p.astype(np.float64) - expect)
    bound = 1e-6 * hp.lr + 2 * U32 * np.abs(expect)
    assert np.all(err <= bound), float(np.max(err / bound))
    # moments after one step: m = (1 - b1) g, v = (1 - b2) g^2
    assert np.allclose(m, 0.1 * g, rtol=3 * U32, atol=0)
    assert np.allclose(v, 0.001 * g * g, rtol=4 * U32, atol=0)


def test_bias_correction_constant_gradient():
    """A constant gradient g for t steps gives m_t = (1 - b1^t) g and
    v_t = (1 - b2^t) g^2, hence m_hat = g, v_hat = g^2 and the same Adam step
    lr * g / (|g| + eps) at every t."""
    hp = oracle.HParams()
    vals = np.array([1e-3, -2.5e-3, 7e-4, -1e-4, 3e-2], np.float32)
    scale = 1024.0
    g_lp = f16(vals * scale)
    g = g_lp.astype(np.float64) / scale
    n = g.size
    p = np.full(n, 0.02, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    sc = oracle.Scaler(loss_scale=scale)
    for t in range(1, 11):
        p_prev = p.astype(np.float64).copy()
        st, _ = step_once(g_lp, "f16", p, m, v, hp, sc)
        assert sc.step == t
        assert np.allclose(m, (1 - hp.beta1 ** t) * g, rtol=t * 4e-7, atol=0)
        assert np.allclose(v, (1 - hp.beta2 ** t) * g * g, rtol=t * 5e-7, atol=0)
        expect = p_prev - hp.lr * (g / (np.abs(g) + hp.eps) + hp.weight_decay * p_prev)
        err = np.abs(p.astype(np.float64) - expect)
        assert np.all(err <= t * 2e-6 * hp.lr + 2 * U32 * np.abs(expect)), (t, err)


def test_decoupled_weight_decay():
    """g = 0: m and v stay 0 and the parameter decays geometrically,
    p_t = p_0 (1 - lr wd)^t.  (L2-style decay folded into g would instead
    make m non-zero and move p by about lr * sign(p) per step.)"""
    hp = oracle.HParams(lr=1e-2, weight_decay=0.1)
    rng = np.random.default_rng(4)
    n = 10000
    p0 = rng.standard_normal(n).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    sc = oracle.Scaler(loss_scale=8.0)
    zero = np.zeros(n, np.float16)
    for t in range(1, 21):
        step_once(zero, "f16", p, m, v, hp, sc)
        assert not m.any() and not v.any()
        expect = p0.astype(np.float64) * (1 - hp.lr * hp.weight_decay) ** t
        assert np.all(np.abs(p - expect) <= t * 3 * U32 * np.abs(expect) + 1e-30)


def textbook(g, p, m, v, t, hp, clip):
    """Kingma & Ba Adam with Loshchilov & Hutter decoupled decay, in binary64
    on binary64 copies of the inputs."""
    g = g * clip
    m1 = hp.beta1 * m + (1 - hp.beta1) * g
    v1 = hp.beta2 * v + (1 - hp.beta2) * g * g
    mh = m1 / (1 - hp.beta1 ** t)
    vh = v1 / (1 - hp.beta2 ** t)
    upd = mh / (np.sqrt(vh) + hp.eps)
    p1 = p - hp.lr * (upd + hp.weight_decay * p)
    return p1, m1, v1, upd


@pytest.mark.parametrize("t0", [0, 1, 4, 99, 4999])
@pytest.mark.parametrize("max_norm", [0.0, 0.05, 100.0])
def test_matches_textbook_binary64(t0, max_norm):
    """The binary32 update against the binary64 textbook formula, within a
    rounding bound derived for the binary32 evaluation: a handful of
    roundings of each term (and of the binary32 step scalars)."""
    rng = np.random.default_rng(5 + t0)
    n = 40000
    scale = 4096.0
    hp = oracle.HParams(max_norm=max_norm)
    g_lp = f16(rng.standard_normal(n).astype(np.float32) * np.float32(1e-3 * scale))
    p = rng.standard_normal(n).astype(np.float32) * np.float32(0.02)
    m = rng.standard_normal(n).astype(np.float32) * np.float32(1e-4)
    v = (np.abs(rng.standard_normal(n)) * 1e-7).astype(np.float32)
    p64, m64, v64 = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    sc = oracle.Scaler(loss_scale=scale, step=t0)
    st, plp = step_once(g_lp, "f16", p, m, v, hp, sc)
    t = t0 + 1
    g = g_lp.astype(np.float64) / scale
    norm = math.sqrt(math.fsum((g * g).tolist()))
    assert abs(st.norm - norm) <= 1e-12 * norm
    clip = 1.0
    if max_norm > 0 and max_norm / (norm + 1e-6) < 1:
        clip = max_norm / (norm + 1e-6)
    # 0.05 is below the norm (about 0.2) and clips; 100 is above it and must not
    assert (clip < 1.0) == (max_norm == 0.05)
    p1, m1, v1, upd = textbook(g, p64, m64, v64, t, hp, clip)
    mterm = np.abs(hp.beta1 * m64) + np.abs((1 - hp.beta1) * g * clip)
    vterm = hp.beta2 * v64 + (1 - hp.beta2) * (g * clip) ** 2
    assert np.all(np.abs(m - m1) <= 4e-7 * mterm + 1e-38)
    assert np.all(np.abs(v - v1) <= 5e-7 * vterm + 1e-38)
    d = np.sqrt(v1 / (1 - hp.beta2 ** t)) + hp.eps
    step_size = hp.lr / (1 - hp.beta1 ** t)
    bound = (step_size * (4e-7 * mterm / d + 1.2e-6 * np.abs(m1) / d)
             + 2 * U32 * np.abs(p1) + 2 * U32 * hp.lr * (np.abs(upd) + hp.weight_decay * np.abs(p64)))
    err = np.abs(p.astype(np.float64) - p1)
    assert np.all(err <= bound), float(np.max(err / bound))
    # the low-precision copy is the master rounded to nearest even
    assert np.array_equal(plp, p.astype(np.float16).view(np.uint16))


def test_matches_torch_adamw():
    """torch.optim.AdamW (CPU, fp32) fed the oracle's unscaled, clipped
    binary32 gradients: a loose, independent cross-check.  At each of 3 steps
    torch starts from the oracle's state, so each step is compared alone
    (torch's own rounding differs and would otherwise accumulate)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    n = 20000
    scale = 1024.0
    hp = oracle.HParams(max_norm=0.05)
    p0 = rng.standard_normal(n).astype(np.float32) * np.float32(0.02)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False)
    sc = oracle.Scaler(loss_scale=scale)
    clipped = 0
    for k in range(3):
        g_lp = f16(rng.standard_normal(n).astype(np.float32) * np.float32(1e-3 * scale))
        p_prev, m_prev, v_prev = p.copy(), m.copy(), v.copy()
        st, _ = step_once(g_lp, "f16", p, m, v, hp, sc)
        g32 = g_lp.astype(np.float32) * np.float32(1 / scale)
        if st.scalars["clip"] != 1.0:
            clipped += 1
            g32 = g32 * np.float32(st.scalars["clip"])
        with torch.no_grad():
            tp.copy_(torch.from_numpy(p_prev))
        if k > 0:
            opt.state[tp]["exp_avg"].copy_(torch.from_numpy(m_prev))
            opt.state[tp]["exp_avg_sq"].copy_(torch.from_numpy(v_prev))
        tp.grad = torch.from_numpy(g32)
        opt.step()
        tm = opt.state[tp]["exp_avg"].numpy()
        tv = opt.state[tp]["exp_avg_sq"].numpy()
        tpp = tp.detach().numpy()
        assert np.all(np.abs(m - tm) <= 1e-6 * (0.9 * np.abs(m_prev) + 0.1 * np.abs(g32)) + 1e-30)
        assert np.all(np.abs(v - tv) <= 1e-6 * (0.999 * v_prev + 0.001 * g32 * g32) + 1e-30)
        assert np.all(np.abs(p - tpp) <= 1e-6 * np.abs(tpp) + 2e-9)
    assert clipped == 3


# ---------------------------------------------------------------- norm, overflow

def test_norm_against_exact_sum():
    rng = np.random.default_rng(7)
    for n in (1, 2, 7, 100, 4097):
        for scale in (1.0, 1024.0, 65536.0):
            g_lp = f16(rng.standard_normal(n).astype(np.float32) * np.float32(1e-3 * scale))
            s, bad = oracle.norm_overflow([g_lp], "f16", scale)
            g = g_lp.astype(np.float64) / scale
            exact = math.fsum((g * g).tolist())  # squares of binary16 values are exact
            assert bad == 0
            assert abs(s - exact) <= n * 2.0 ** -53 * exact


def test_norm_closed_forms():
    # all-equal gradients c: norm = |c| sqrt(n); exact for c, n powers of two
    for k in (0, 5, 12):
        n = 1 << k
        g = np.full(n, 0.5, np.float16)
        s, _ = oracle.norm_overflow([g], "f16", 1.0)
        assert s == 0.25 * n
        assert math.sqrt(s) == 0.5 * math.sqrt(n)
    # unscaling by a power of two is exact: S * g with 1/S equals g with 1
    rng = np.random.default_rng(8)
    g = f16(rng.standard_normal(1000) * 1e-2)
    base, _ = oracle.norm_overflow([g], "f16", 1.0)
    for S in (2.0, 256.0, 4096.0):
        gs = f16(g.astype(np.float32) * np.float32(S))
        assert np.array_equal(gs.astype(np.float32), g.astype(np.float32) * np.float32(S))
        s, _ = oracle.norm_overflow([gs], "f16", S)
        assert s == base
    # folding several arrays equals one concatenated array (same order)
    parts = [f16(rng.standard_normal(n) * 1e-2) for n in (3, 100, 1, 57)]
    s_parts, _ = oracle.norm_overflow(parts, "f16", 1.0)
    s_cat, _ = oracle.norm_overflow([np.concatenate(parts)], "f16", 1.0)
    assert s_parts == s_cat


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("where", ["first", "middle", "last"])
@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_overflow_detection(dtype, where, bad):
    n = 1001
    x = np.random.default_rng(9).standard_normal(n).astype(np.float32) * np.float32(1e-2)
    i = {"first": 0, "middle": n // 2, "last": n - 1}[where]
    x[i] = bad
    g = zs.host_cast(x, dtype)
    _, flag = oracle.norm_overflow([g], dtype, 1.0)
    assert flag == 1
    x[i] = 0.0
    _, flag = oracle.norm_overflow([zs.host_cast(x, dtype)], dtype, 1.0)
    assert flag == 0
    # the largest finite binary16 is not an overflow
    big = np.full(4, 65504.0, np.float16)
    assert oracle.norm_overflow([big], "f16", 1.0)[1] == 0


def test_skip_leaves_state_untouched_and_halves_scale():
    rng = np.random.default_rng(10)
    n = 5000
    p = rng.standard_normal(n).astype(np.float32)
    m = rng.standard_normal(n).astype(np.float32) * np.float32(1e-4)
    v = np.abs(rng.standard_normal(n)).astype(np.float32) * np.float32(1e-7)
    plp = rng.integers(0, 65535, n).astype(np.uint16)
    before = [a.copy() for a in (p, m, v, plp)]
    g = f16(rng.standard_normal(n) * 10)
    g[1234] = np.inf
    hp = oracle.HParams(max_norm=1.0)
    sc = oracle.Scaler(loss_scale=65536.0, step=7, good_steps=5)
    st = oracle.adam_step([g], "f16", [p], [m], [v], [plp], "f16", hp, sc)
    assert st.skip
    for a, b in zip((p, m, v, plp), before):
        assert a.tobytes() == b.tobytes()
    assert sc.loss_scale == 32768.0 and sc.step == 7 and sc.good_steps == 0
    # the floor holds
    sc = oracle.Scaler(loss_scale=1.0, step=3)
    oracle.adam_step([g], "f16", [p], [m], [v], [plp], "f16", hp, sc)
    assert sc.loss_scale == 1.0 and sc.step == 3


def test_scale_growth_after_window():
    hp = oracle.HParams(scale_window=3)
    sc = oracle.Scaler(loss_scale=8.0)
    n = 64
    p, m, v = np.ones(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    g = np.full(n, 0.25, np.float16)
    scales = []
    for _ in range(7):
        oracle.adam_step([g], "f16", [p], [m], [v], [None], "f16", hp, sc)
        scales.append(sc.loss_scale)
    assert scales == [8.0, 8.0, 16.0, 16.0, 16.0, 32.0, 32.0]
    assert sc.step == 7


# ---------------------------------------------------------------- accumulate

def test_accumulate_order_and_exactness():
    # micro-batch order k = 0..3 fixes the rounding: 1 + 2^-24 + 2^-24 + 0
    # is 1 in binary32 (two ties to even); the reverse order gives 1 + 2^-23
    bufs = [zs.host_cast(np.array([v], np.float32), "bf16") for v in (1.0, 2.0 ** -24, 2.0 ** -24, 0.0)]
    acc = np.zeros(1, np.float32)
    oracle.accumulate(acc, bufs, "bf16", overwrite=True)
    assert acc[0] == np.float32(1.0)
    acc2 = np.zeros(1, np.float32)
    oracle.accumulate(acc2, bufs[::-1], "bf16", overwrite=True)
    assert acc2[0] == np.float32(1.0) + np.float32(2.0 ** -23)
    # integer-valued micro-batch gradients sum exactly
    rng = np.random.default_rng(11)
    ints = [rng.integers(-100, 100, 999).astype(np.float32) for _ in range(4)]
    acc = np.full(999, 5.0, np.float32)
    oracle.accumulate(acc, [zs.host_cast(x, "bf16") for x in ints], "bf16", overwrite=False)
    assert np.array_equal(acc, 5.0 + sum(ints))
    oracle.accumulate(acc, [zs.host_cast(x, "f16") for x in ints], "f16", overwrite=True)
    assert np.array_equal(acc, sum(ints))


# ---------------------------------------------------------------- partition invariance

@pytest.mark.parametrize("max_norm", [0.0, 0.5])
def test_partition_invariance(max_norm):
    """The Nd shards of the flat partition, updated with the global norm and
    overflow, concatenate to the unpartitioned update, bit for bit."""
    numel = zs.numels(zs.tiny_transformer_shapes(hidden=32, vocab=64))
    nd, align = 4, 8
    lay = oracle.partition_layout(numel, nd, align)
    total = sum(numel)
    hp = oracle.HParams(max_norm=max_norm)
    p0 = np.zeros(lay.padded_total, np.float32)
    p0[:total] = zs.host_master(total, 0)
    flat = [p0.copy(), np.zeros_like(p0), np.zeros_like(p0), np.zeros(lay.padded_total, np.uint16)]
    S = lay.shard_numel
    shards = [[a[r * S:(r + 1) * S].copy() for a in flat] for r in range(nd)]
    sc_a, sc_b = oracle.Scaler(loss_scale=1024.0), oracle.Scaler(loss_scale=1024.0)
    for step in range(3):
        g = np.zeros(lay.padded_total, np.float16)
        g[:total] = zs.host_grad(total, 0, step, 1024.0, "f16")
        oracle.adam_step([g], "f16", [flat[0]], [flat[1]], [flat[2]], [flat[3]], "f16", hp, sc_a)
        oracle.adam_step([g[r * S:(r + 1) * S].copy() for r in range(nd)], "f16",
                         [s[0] for s in shards], [s[1] for s in shards], [s[2] for s in shards],
                         [s[3] for s in shards], "f16", hp, sc_b)
    for k in range(4):
        cat = np.concatenate([s[k] for s in shards])
        assert cat.tobytes() == flat[k].tobytes()
    # the zero padding stays exactly zero
    assert not flat[0][total:].any() and not flat[1][total:].any() and not flat[2][total:].any()


# ---------------------------------------------------------------- memory arithmetic

def test_memory_arithmetic_matches_pages():
    import json, os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "memory_pages.json")))
    a = gold["state_1p5b"]
    assert oracle.model_state_bytes(int(a["params"])) == a["min_state_bytes"]
    b = gold["fp16_weights_1p5b"]
    assert b["params"] * oracle.BYTES_PER_PARAM["p16"] == b["approx_bytes"]
    c = gold["state_1t"]
    total = oracle.model_state_bytes(int(c["params"]))
    assert total == c["approx_total_bytes"]
    per_gpu = oracle.model_state_bytes(int(c["params"]), nd=c["gpus"], stage=3)
    assert abs(per_gpu - c["approx_bytes_per_gpu"]) / c["approx_bytes_per_gpu"] < 0.03
    assert per_gpu < c["gpu_memory_bytes"]
    r = gold["stage_reduction"]
    psi = 10 ** 9
    base = oracle.model_state_bytes(psi)
    for stage, cut in ((1, r["stage1"]), (2, r["stage2"])):
        ratio = base / oracle.model_state_bytes(psi, nd=4096, stage=stage)
        assert abs(ratio - cut) / cut < 0.01
        assert base / oracle.model_state_bytes(psi, nd=1, stage=stage) == 1.0
    for nd in (2, 16, 400):
        assert base / oracle.model_state_bytes(psi, nd=nd, stage=3) == nd
    d = gold["config_100b"]
    assert d["gpus"] % d["model_parallel"] == 0
    dp = d["gpus"] // d["model_parallel"]
    h = d["hidden"]
    stack = zs.numels(zs.layer_stack_shapes(d["layers"], h))
    assert sum(stack) == d["layers"] * (12 * h * h + 13 * h)
    # one model-parallel slice of the 100B model spread over the DP ranks
    # under stage 2 fits a 32 GB V100 (derived, not printed)
    psi_mp = sum(stack) / d["model_parallel"]
    assert oracle.model_state_bytes(psi_mp, nd=dp, stage=2) < 32e9


# ---------------------------------------------------------------- stage-2 reduction

def test_reduce_mean_closed_forms():
    from fractions import Fraction
    rng = np.random.default_rng(12)
    x = f16(rng.standard_normal(5000) * 3)
    # equal replicas: the mean is the value itself, for any count
    for k in (1, 2, 3, 7, 16):
        out = oracle.reduce_mean([x] * k, "f16", "f16")
        assert np.array_equal(out, x.view(np.uint16))
    # power-of-two counts: sum exact (integers), division exact
    ints = [rng.integers(-200, 200, 999).astype(np.float32) for _ in range(8)]
    out = oracle.reduce_mean([zs.host_cast(a, "bf16") for a in ints], "bf16", "f32")
    assert np.array_equal(out, sum(ints) / np.float32(8))
    # three replicas: the correctly rounded binary32 quotient of the exact
    # integer sum by 3 (a reciprocal multiply rounds some of these the other way)
    sums = np.arange(1, 20001, dtype=np.int64)
    a = [np.zeros(sums.size, np.float32), np.zeros(sums.size, np.float32), sums.astype(np.float32)]
    out = oracle.reduce_mean(a, "f32", "f32")
    exact = np.array([float(Fraction(int(t), 3)) for t in sums]).astype(np.float32)
    assert np.array_equal(out, exact)
    recip = (sums.astype(np.float32) * np.float32(1 / 3)).astype(np.float32)
    assert not np.array_equal(out, recip)  # the pin distinguishes the two
    # rank order fixes the rounding: 1 + 2^-24 + 2^-24 + 0 stays 1 (two ties)
    r = [np.array([v], np.float32) for v in (1.0, 2.0 ** -24, 2.0 ** -24, 0.0)]
    assert oracle.reduce_mean(r, "f32", "f32")[0] == np.float32(0.25)
    assert oracle.reduce_mean(r[::-1], "f32", "f32")[0] == (np.float32(1.0) + np.float32(2.0 ** -23)) / 4
    # an inf in any replica reaches the output
    y = x.copy()
    y[10] = np.inf
    out = oracle.reduce_mean([x, y, x], "f16", "f16").view(np.float16)
    assert np.isinf(out[10]) and np.isfinite(out[11])


# ---------------------------------------------------------------- helpers the GPU tests use

@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "f16")])
def test_adam_apply_sampled_equals_whole_update_gathered(gdtype, pdtype):
    """The sampled update (state arrays holding only the sampled elements)
    against the whole-array update gathered at the samples: equal bit for
    bit over three steps, for samples that include both ends, repeats and an
    unsorted order."""
    rng = np.random.default_rng(21)
    n = 10_007
    scale = 1.0 if gdtype == "bf16" else 1024.0
    idx = np.concatenate([[0, n - 1, 5, 5], rng.integers(0, n, 500)]).astype(np.int64)
    rng.shuffle(idx)
    p = zs.host_master(n, 3)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    plp = np.zeros(n, np.uint16)
    ps, ms, vs, plps = p[idx].copy(), m[idx].copy(), v[idx].copy(), np.zeros(idx.size, np.uint16)
    hp = oracle.HParams(max_norm=0.05)
    sc = oracle.Scaler(loss_scale=scale)
    for k in range(3):
        g = zs.host_grad(n, 3, k, scale, gdtype)
        sumsq, bad = oracle.norm_overflow([g], gdtype, scale)
        st = oracle.decide(hp, sc, sumsq, bad)
        oracle.adam_apply(g, gdtype, p, m, v, plp, pdtype, st)
        oracle.adam_apply_sampled(g, gdtype, idx, ps, ms, vs, plps, pdtype, st)
        for name, whole, sampled in (("p", p, ps), ("m", m, ms), ("v", v, vs), ("p_lp", plp, plps)):
            assert whole[idx].tobytes() == sampled.tobytes(), f"{name} step {k}"
    assert sc.step == 3 and st.scalars["clip"] < 1.0


def test_with_clip_changes_only_the_clip_coefficient():
    """with_clip(step, c) is the step with c as its binary32 clip
    coefficient and nothing else changed: with c = 1/2 it updates exactly as
    the unclipped step does on gradients halved beforehand (both products
    are exact for these normal values), and with the step's own coefficient
    it is the same step."""
    rng = np.random.default_rng(22)
    n = 4096
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    hp, sc = oracle.HParams(), oracle.Scaler(loss_scale=1.0)
    st = oracle.decide(hp, sc, float(np.sum(g.astype(np.float64) ** 2)), 0)
    assert st.scalars["clip"] == 1.0
    half = oracle.with_clip(st, 0.5)
    assert half.scalars["clip"] == 0.5 and half.skip == st.skip and half.norm == st.norm
    assert {k: x for k, x in half.scalars.items() if k != "clip"} == \
           {k: x for k, x in st.scalars.items() if k != "clip"}
    p0 = zs.host_master(n, 4)
    runs = []
    for step, grad in ((half, g), (st, g * np.float32(0.5)), (oracle.with_clip(st, 1.0), g * np.float32(0.5))):
        p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        oracle.adam_apply(grad, "f32", p, m, v, None, "f16", step)
        runs.append((p, m, v))
    for a, b in zip(runs[0], runs[1]):
        assert a.tobytes() == b.tobytes()
    for a, b in zip(runs[1], runs[2]):
        assert a.tobytes() == b.tobytes()
    # and it is not the unclipped update
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam_apply(g, "f32", p, m, v, None, "f16", st)
    assert m.tobytes() != runs[0][1].tobytes()
