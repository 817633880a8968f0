"""The pins must be able to fail: each test here builds a copy of the oracle's
C source with one plausible mistake planted in it (CPU only, in a temporary
directory), swaps it in, and checks that at least one pin rejects it."""
import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "zero_oracle.c")

# (name, text in the source, replacement)
MUTANTS = [
    ("decay sign", "- (s->step_size * u + s->lr_wd * *p)", "- (s->step_size * u - s->lr_wd * *p)"),
    ("decay dropped", "- (s->step_size * u + s->lr_wd * *p)", "- (s->step_size * u)"),
    ("bias correction one step late", "pow(hp->beta1, t)", "pow(hp->beta1, t + 1.0)"),
    ("beta1 in second correction", "pow(hp->beta2, t)", "pow(hp->beta1, t)"),
    ("second correction dropped", "(float)(1.0 / sqrt(bc2))", "1.0f"),
    ("first correction dropped", "(float)(hp->lr / bc1)", "(float)hp->lr"),
    ("eps inside the root", "sqrtf(v1) * s->inv_sqrt_bc2 + s->eps", "sqrtf(v1 + s->eps) * s->inv_sqrt_bc2"),
    ("moment coefficients swapped", "s->beta1 * *m + s->one_minus_beta1 * g",
     "s->one_minus_beta1 * *m + s->beta1 * g"),
    ("variance takes 1-b1", "s->one_minus_beta2 * (g * g)", "s->one_minus_beta1 * (g * g)"),
    ("variance of |g| not g^2", "s->one_minus_beta2 * (g * g)", "s->one_minus_beta2 * fabsf(g)"),
    ("unscale dropped in update", "float g = g_lp * s->inv_scale;", "float g = g_lp;"),
    ("skip ignored", "    if (s->skip)\n        return;\n    for (int64_t i = 0; i < n; ++i) {\n        adam_element",
     "    for (int64_t i = 0; i < n; ++i) {\n        adam_element"),
    ("scale doubled on overflow", "double s = sc->loss_scale / 2.0;", "double s = sc->loss_scale * 2.0;"),
    ("step counted on skip", "        sc->good_steps = 0;\n        out->clip = 1.0f;",
     "        sc->good_steps = 0;\n        sc->step += 1;\n        out->clip = 1.0f;"),
    ("clip above one", "if (c < 1.0)", "if (c > 0.0)"),
    ("norm of scaled gradient", "float gi = load_elem(g, dtype, i) * inv_scale;",
     "float gi = load_elem(g, dtype, i);"),
    ("overflow test dropped", "if (!isfinite(gi))\n            bad = 1;", ""),
    ("growth window off by one", "if (sc->good_steps >= hp->scale_window)",
     "if (sc->good_steps > hp->scale_window)"),
    ("accumulation reversed", "for (; k < n_bufs; ++k)\n            a = a + load_elem(bufs[k], dtype, i);",
     "for (int32_t j = n_bufs - 1; j >= k; --j)\n            a = a + load_elem(bufs[j], dtype, i);"),
    ("bf16 ties away", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("f16 truncation", "_Float16 h = (_Float16)x;", "_Float16 h = (_Float16)(x - x * 0x1p-12f);"),
    ("mean by reciprocal", "const float mean = a / count;", "const float mean = a * (1.0f / count);"),
    ("mean over one replica fewer", "const float count = (float)n_bufs;",
     "const float count = (float)(n_bufs > 1 ? n_bufs - 1 : 1);"),
    ("sampled update reads the gradient at the sample's position",
     "adam_element(load_elem(g, gdtype, idx[j]), &p[j]", "adam_element(load_elem(g, gdtype, j), &p[j]"),
    ("reduction reversed", "        float a = load_elem(bufs[0], dtype, i);\n        for (int32_t k = 1; k < n_bufs; ++k)\n            a = a + load_elem(bufs[k], dtype, i);",
     "        float a = load_elem(bufs[n_bufs - 1], dtype, i);\n        for (int32_t k = n_bufs - 2; k >= 0; --k)\n            a = a + load_elem(bufs[k], dtype, i);"),
]

PINS = [
    pins.test_f16_cast_matches_numpy,
    pins.test_bf16_cast_matches_torch,
    lambda: pins.test_step1_closed_form(0.0),
    lambda: pins.test_step1_closed_form(1e-8),
    pins.test_bias_correction_constant_gradient,
    pins.test_decoupled_weight_decay,
    lambda: pins.test_matches_textbook_binary64(4, 0.0),
    lambda: pins.test_matches_textbook_binary64(0, 0.05),
    lambda: pins.test_matches_textbook_binary64(1, 100.0),
    pins.test_matches_torch_adamw,
    pins.test_norm_against_exact_sum,
    pins.test_norm_closed_forms,
    lambda: pins.test_overflow_detection("f16", "middle", float("inf")),
    pins.test_skip_leaves_state_untouched_and_halves_scale,
    pins.test_scale_growth_after_window,
    pins.test_accumulate_order_and_exactness,
    pins.test_reduce_mean_closed_forms,
    lambda: pins.test_adam_apply_sampled_equals_whole_update_gathered("f16", "f16"),
]


def run_pins() -> list[str]:
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError) as e:
            failed.append(f"{getattr(pin, '__name__', 'pin')}: {type(e).__name__}")
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique for {name!r}"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = oracle.compile_source(str(mutant_src), str(tmp_path / "libmutant.so"))
    saved = oracle._lib
    oracle._lib = oracle.load(so)
    try:
        failed = run_pins()
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_oracle_passes_every_pin():
    assert run_pins() == []
