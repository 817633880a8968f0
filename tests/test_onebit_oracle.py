"""Pins for the oracle's 1-bit Adam compression stage (CPU only).

The pages name 1-bit Adam without its algorithm, so these pins check the
oracle against mathematics, not against printed numbers: the compressor's
closed forms (constant magnitudes, zeros, the L2 scale), the error-feedback
identity at both ends of the compressed all-reduce within a derived rounding
bound, the server's average against exact rational arithmetic, the frozen
variance against the warm-up's own decision, and a whole step whose
compression is exact against a binary64 evaluation.  Planted mistakes in the
C source and the Python layer must each fail a pin."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import zero_synth as zs

F32 = np.float32


def _hp(**kw):
    return oracle.HParams(**kw)


def _compress_step():
    """Step scalars with beta1 = 0 and loss scale 1: the worker's local
    momentum is then the fp32 'gradient' itself, so the worker call is the
    compressor applied to x + e."""
    return oracle.decide(_hp(beta1=0.0), oracle.Scaler(loss_scale=1.0), 0.0, 0)


def compress(x, e, x_out=None):
    """C(x + e) through the worker: returns (bits, scale); e updated (and
    x_out, if given, holds the compressed value x + e)."""
    m = np.zeros(x.size, F32)
    return oracle.onebit_worker(np.ascontiguousarray(x, F32), "f32", _compress_step(), m, e, x_out=x_out)


def unpack(bits, n):
    """Element k's sign bit, decoded independently of the oracle (numpy's
    little-endian bit order over the little-endian words)."""
    u8 = np.ascontiguousarray(bits, dtype="<u4").view(np.uint8)
    return np.unpackbits(u8, bitorder="little")[:n].astype(bool)


# ---------------------------------------------------------------- the compressor

@pytest.mark.parametrize("n", [1, 31, 32, 1000, 1001])
def test_compress_constant_magnitude_is_exact(n):
    rng = np.random.default_rng(n)
    c = F32(0.375)
    signs = rng.integers(0, 2, n).astype(bool)
    x = np.where(signs, c, -c).astype(F32)
    e = np.zeros(n, F32)
    bits, scale = compress(x, e)
    assert scale == c
    assert not e.any()
    assert np.array_equal(unpack(bits, n), signs)


def test_compress_zeros_and_signed_zero():
    x = np.array([0.0, -0.0, 0.0, -0.0] * 10, F32)
    e = np.zeros(x.size, F32)
    bits, scale = compress(x, e)
    assert scale == 0.0
    assert unpack(bits, x.size).all()  # sign(0) = sign(-0) = +1
    assert not e.any()


@pytest.mark.parametrize("n", [1, 33, 4096, 10_007])
def test_compress_scale_is_the_l2_scale_and_signs_are_bits(n):
    rng = np.random.default_rng(10 + n)
    x = (rng.standard_normal(n) * 1e-3).astype(F32)
    e0 = (rng.standard_normal(n) * 1e-4).astype(F32)
    buf = (x + e0).astype(F32)  # the binary32 sum the compressor sees
    e = e0.copy()
    seen = np.full(n, np.nan, F32)
    bits, scale = compress(x, e, seen)
    # the compressor's input as reported is the binary32 sum itself
    assert seen.tobytes() == buf.tobytes()
    exact = math.sqrt(math.fsum(float(b) * float(b) for b in buf) / n)
    assert abs(scale - exact) <= 2.0 ** -24 * exact * (1 + 1e-9)
    assert np.array_equal(unpack(bits, n), ~(buf < 0))
    # the new error is buf - scale*sign, one rounding
    want = np.where(buf < 0, buf + F32(scale), buf - F32(scale)).astype(F32)
    assert np.array_equal(e, want)


def _feedback_bound(bufs, errs):
    return sum((np.abs(b.astype(np.float64)) + np.abs(r.astype(np.float64))) for b, r in
               zip(bufs, errs)) * 2.0 ** -24


def test_worker_error_feedback_telescopes():
    """sum_t C_t + e_T = sum_t x_t up to the two binary32 roundings a step."""
    rng = np.random.default_rng(3)
    n, T = 777, 25
    e = np.zeros(n, F32)
    sum_x, sum_c = np.zeros(n), np.zeros(n)
    bufs, errs = [], []
    for t in range(T):
        x = (rng.standard_normal(n) * (1 + t % 3)).astype(F32)
        bufs.append((x + e).astype(F32))
        bits, scale = compress(x, e)
        errs.append(e.copy())
        sgn = np.where(unpack(bits, n), 1.0, -1.0)
        sum_x += x
        sum_c += sgn * scale
    gap = np.abs(sum_c + e.astype(np.float64) - sum_x)
    assert (gap <= _feedback_bound(bufs, errs) * 1.01 + 1e-300).all()
    # and the feedback is doing something: the error stays bounded by the
    # scales rather than growing with T
    assert np.abs(e).max() < 4 * max(np.abs(b).max() for b in bufs)


def test_worker_local_momentum_without_gradient():
    """g = 0: the local momentum is b1*m; for m = +-c it has the one
    magnitude f32(b1*c), so the compression is exact and gives it back."""
    n = 640
    rng = np.random.default_rng(21)
    c = F32(0.5)
    signs = rng.integers(0, 2, n).astype(bool)
    m = np.where(signs, c, -c).astype(F32)
    e = np.zeros(n, F32)
    hp = _hp()
    st = oracle.decide(hp, oracle.Scaler(loss_scale=1.0), 0.0, 0)
    bits, scale = oracle.onebit_worker(np.zeros(n, np.float16), "f16", st, m, e)
    assert scale == F32(F32(hp.beta1) * c)
    assert np.array_equal(unpack(bits, n), signs) and not e.any()


# ---------------------------------------------------------------- the server

@pytest.mark.parametrize("nd", [1, 2, 3, 5, 16])
def test_server_average_is_the_correctly_rounded_mean(nd):
    rng = np.random.default_rng(40 + nd)
    S = 320
    scales = [F32(int(k) / 64) for k in rng.integers(1, 200, nd)]
    bits = [rng.integers(0, 2 ** 32, S // 32, dtype=np.uint32) for _ in range(nd)]
    f = np.zeros(S, F32)
    # a forced scale of 0 leaves f' = y exactly (y - 0*sign)
    oracle.onebit_server(bits, scales, f, scale=0.0)
    for i in range(S):
        q = sum(Fraction(float(scales[k])) * (1 if (bits[k][i // 32] >> (i % 32)) & 1 else -1)
                for k in range(nd)) / nd
        y = f[i]
        for nb in (np.nextafter(y, F32(np.inf)), np.nextafter(y, F32(-np.inf))):
            assert abs(Fraction(float(y)) - q) <= abs(Fraction(float(nb)) - q)


def test_server_sum_runs_in_rank_order():
    """The workers' terms are added in rank order, starting from worker 0's
    term: with scales 1, 2^-24, 2^-24 and every sign +, 1 + 2^-24 is a tie
    that rounds to 1, twice, so the mean is binary32(1/3); the reverse order
    (2^-24 + 2^-24 = 2^-23 exactly, then 1 + 2^-23 exactly) would give
    binary32((1 + 2^-23)/3), one ulp above.  With worker 0's sign -, the
    first addition -1 + 2^-24 is exact (1 - 2^-24 is a binary32 value) and
    so is the second: the mean is binary32((-1 + 2^-23)/3)."""
    S = 64
    scales = [F32(1.0), F32(2.0 ** -24), F32(2.0 ** -24)]
    plus = [np.full(S // 32, 0xFFFFFFFF, np.uint32) for _ in range(3)]
    f = np.zeros(S, F32)
    oracle.onebit_server(plus, scales, f, scale=0.0)
    third = F32(F32(1.0) / F32(3.0))
    assert (f == third).all()
    assert third != F32(float(Fraction(1) + Fraction(1, 2 ** 23)) / 3.0)
    minus0 = [np.zeros(S // 32, np.uint32)] + plus[1:]
    f = np.zeros(S, F32)
    oracle.onebit_server(minus0, scales, f, scale=0.0)
    want = F32(float(Fraction(-1) + Fraction(1, 2 ** 23))) / F32(3.0)
    assert (f == want).all()


def test_server_error_feedback_telescopes():
    rng = np.random.default_rng(9)
    S, nd, T = 640, 4, 20
    f = np.zeros(S, F32)
    sum_y, sum_s = np.zeros(S), np.zeros(S)
    bufs, errs = [], []
    for t in range(T):
        scales = [F32(x) for x in rng.uniform(0.5, 2.0, nd)]
        bits = [rng.integers(0, 2 ** 32, S // 32, dtype=np.uint32) for _ in range(nd)]
        avg = np.zeros(S, F32)
        oracle.onebit_server(bits, scales, avg, scale=0.0)  # avg alone
        bufs.append((avg + f).astype(F32))
        out_bits, s = oracle.onebit_server(bits, scales, f)
        errs.append(f.copy())
        sum_y += avg
        sum_s += np.where(unpack(out_bits, S), 1.0, -1.0) * s
    gap = np.abs(sum_s + f.astype(np.float64) - sum_y)
    assert (gap <= _feedback_bound(bufs, errs) * 1.01).all()


# ---------------------------------------------------------------- the step

def test_variance_correction_frozen_at_the_last_warmup_step():
    hp = _hp()
    T = 50
    sc = oracle.Scaler(loss_scale=1.0, step=T - 1)
    warm = oracle.decide(hp, sc, 0.0, 0)  # the decision of warm-up step T
    assert sc.step == T
    for k in range(1, 6):
        st = oracle.frozen_variance(oracle.decide(hp, sc, 0.0, 0), hp, T)
        plain = oracle.decide(hp, oracle.Scaler(loss_scale=1.0, step=T + k - 1), 0.0, 0)
        assert st.scalars["inv_sqrt_bc2"] == warm.scalars["inv_sqrt_bc2"]
        assert st.scalars["step_size"] == plain.scalars["step_size"]


@pytest.mark.parametrize("nd", [1, 2, 4, 16])
def test_whole_step_with_exact_compression_matches_binary64(nd):
    """Every worker sees the same gradient +-c and m = e = 0; with
    1 - b1 = 1/8 the local momenta are +-a, a = c/8 (a power of two), so both
    compressions are exact (the server's partial sums k*a and the division by
    a power-of-two Nd are exact too), the synchronised momentum is +-a, the
    errors stay 0, and the update is
    p - lr/(1-b1^t) * m/(sqrt(v/(1-b2^T)) + eps) - lr*wd*p in binary64 up
    to the binary32 roundings."""
    S = 256
    n, numel = nd * S, nd * S - 7
    rng = np.random.default_rng(nd)
    c, scale = 0.25, 1024.0
    signs = rng.integers(0, 2, n).astype(bool)
    g = np.where(signs, c * scale, -c * scale).astype(np.float16)
    grads = [g.copy() for _ in range(nd)]
    p = zs.host_master(n, 1)
    p0 = p.copy()
    m = np.zeros(n, F32)
    v = (rng.uniform(0.5, 2.0, n) * 1e-6).astype(F32)
    ew = [np.zeros(n, F32) for _ in range(nd)]
    es = [np.zeros(S, F32) for _ in range(nd)]
    hp, T = _hp(beta1=0.875), 40
    sc = oracle.Scaler(loss_scale=scale, step=T)
    res = oracle.onebit_step(grads, "f16", S, numel, p, m, v, ew, es, None, "f16", hp, sc, T)
    a = F32(c / 8)
    assert all(s == a for s in res.worker_scales) and all(s == a for s in res.server_scales)
    assert not any(e.any() for e in ew) and not any(e.any() for e in es)
    t = T + 1
    mh = np.where(signs, float(a), -float(a))
    vh = v.astype(np.float64) / (1 - hp.beta2 ** T)
    step = hp.lr / (1 - hp.beta1 ** t) * mh / (np.sqrt(vh) + hp.eps)
    decay = hp.lr * hp.weight_decay * p0
    want = p0 - step - decay
    got = p.astype(np.float64)
    # a handful of binary32 roundings, each within half an ulp of a value no
    # larger than |p| + |step| + |decay|
    bound = 8 * 2.0 ** -24 * (np.abs(p0) + np.abs(step) + np.abs(decay))
    assert (np.abs(got - want)[:numel] <= bound[:numel]).all()
    # the padding beyond numel is not parameters: untouched; the momentum
    # covers the whole padded buffer
    assert np.array_equal(p[numel:], p0[numel:])
    assert np.array_equal(m, np.where(signs, a, -a))


def test_skipped_step_changes_nothing():
    nd, S = 2, 128
    n = nd * S
    grads = [zs.host_grad(n, i, 0, 1024.0, "f16") for i in range(nd)]
    grads[1][77] = np.float16(np.inf)
    p = zs.host_master(n, 0)
    m = np.full(n, F32(1e-4))
    v = np.full(n, F32(1e-6))
    ew = [np.full(n, F32(1e-5)) for _ in range(nd)]
    es = [np.full(S, F32(2e-5)) for _ in range(nd)]
    before = [a.tobytes() for a in [p, m, v] + ew + es]
    sc = oracle.Scaler(loss_scale=1024.0, step=10)
    res = oracle.onebit_step(grads, "f16", S, n, p, m, v, ew, es, None, "f16", _hp(), sc, 10)
    assert res.step.skip and sc.step == 10 and sc.loss_scale == 512.0
    assert [a.tobytes() for a in [p, m, v] + ew + es] == before


def test_comm_ratio_closed_forms():
    assert oracle.onebit_comm_ratio(0.0) == 32.0
    assert oracle.onebit_comm_ratio(1.0) == 1.0


# ---------------------------------------------------------------- the pins can fail

PINS = [
    lambda: [test_compress_constant_magnitude_is_exact(n) for n in (1, 31, 32, 1000, 1001)],
    test_compress_zeros_and_signed_zero,
    lambda: [test_compress_scale_is_the_l2_scale_and_signs_are_bits(n) for n in (1, 33, 4096)],
    test_worker_error_feedback_telescopes,
    test_worker_local_momentum_without_gradient,
    lambda: [test_server_average_is_the_correctly_rounded_mean(nd) for nd in (1, 2, 3, 5)],
    test_server_sum_runs_in_rank_order,
    test_server_error_feedback_telescopes,
    test_variance_correction_frozen_at_the_last_warmup_step,
    lambda: [test_whole_step_with_exact_compression_matches_binary64(nd) for nd in (1, 2, 4)],
    test_skipped_step_changes_nothing,
]

SRC = os.path.join(os.path.dirname(oracle.__file__), "zero_oracle.c")

C_MUTANTS = [
    ("sign of zero negative", "const int plus = !(buf[i] < 0.0f);", "const int plus = buf[i] > 0.0f;"),
    ("scale over n - 1", "sqrt(s / (double)n)", "sqrt(s / (double)(n > 1 ? n - 1 : 1))"),
    ("worker error feedback dropped", "e[i] = mi + e[i];", "e[i] = mi;"),
    ("error not kept", "buf[i] = buf[i] - (plus ? sc : -sc);", "buf[i] = 0.0f * buf[i];"),
    ("error sign flipped", "buf[i] = buf[i] - (plus ? sc : -sc);", "buf[i] = (plus ? sc : -sc) - buf[i];"),
    ("bits big-endian", "bits[i / 32] |= 1u << (i % 32);", "bits[i / 32] |= 1u << (31 - i % 32);"),
    ("compressor input not reported", "    if (x_out)\n", "    if (x_out && n < 0)\n"),
    ("server mean over nd - 1", "const float count = (float)nd;",
     "const float count = (float)(nd > 1 ? nd - 1 : 1);"),
    ("server error feedback dropped", "f[i] = a / count + f[i];", "f[i] = a / count;"),
    ("server sum in reverse rank order",
     "for (int32_t k = 0; k < nd; ++k) {\n            const float c = ((bits[k][i / 32] >> (i % 32)) & 1u) ? "
     "scales[k] : -scales[k];\n            a = k == 0 ? c : a + c;",
     "for (int32_t k = nd - 1; k >= 0; --k) {\n            const float c = ((bits[k][i / 32] >> (i % 32)) & 1u) ? "
     "scales[k] : -scales[k];\n            a = k == nd - 1 ? c : a + c;"),
    ("momentum not synchronised", "        m[i] = mi;\n        if (i >= numel)", "        if (i >= numel)"),
    ("local momentum drops beta1", "const float mi = s->beta1 * m[i] + s->one_minus_beta1 * gi;",
     "const float mi = s->one_minus_beta1 * gi;"),
]

PY_MUTANTS = [
    ("frozen_variance", "hp.beta2 ** float(t_freeze)", "hp.beta2 ** float(t_freeze + 1)"),
]


def run_pins():
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError) as e:
            failed.append(f"{getattr(pin, '__name__', 'pin')}: {type(e).__name__}")
    return failed


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_planted_c_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique for {name!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    saved = oracle._lib
    oracle._lib = oracle.load(so)
    try:
        failed = run_pins()
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake {name!r}"


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_python_mistake_is_caught(name, old, new, monkeypatch):
    import inspect
    src = inspect.getsource(getattr(oracle, name))
    assert old in src
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, name, ns[name])
    assert run_pins(), f"no pin caught the planted mistake in {name}"


def test_unmutated_oracle_passes_every_pin():
    assert run_pins() == []
