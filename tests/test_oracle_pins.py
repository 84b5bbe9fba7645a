"""The oracle against facts the definition fixes (closed forms, invariants, brute force, the worked example).

Also checks that the pins have teeth: each plausible mistake, planted in a copy of
the oracle's C source built in a temporary directory, fails at least one pin that
does not lean on the oracle's own long-double brute force.
"""

import os

import numpy as np
import pytest

import oracle
import pins
import synth


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_shape_convention():
    pins.pin_shape_convention()


def test_generator_matches_published_splitmix64():
    # First outputs of Vigna's splitmix64.c seeded with 0.
    z = synth.splitmix64(0, 0, 3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generator_slices_are_consistent():
    a = synth.splitmix64(7, 0, 100)
    b = synth.splitmix64(7, 40, 20)
    assert np.array_equal(a[40:60], b)
    q1 = synth.make_qkv(1, 2, 33, 17, 8, 8, "bf16", seed=5)
    q2 = synth.make_qkv(1, 2, 33, 17, 8, 8, "bf16", seed=5)
    assert all(np.array_equal(x, y) for x, y in zip(q1, q2))


def test_generator_distributions():
    x = synth.normal(3, 0, 200000, sigma=4.0)
    assert abs(x.mean()) < 0.05 and abs(x.std() - 4.0) < 0.05
    u = 2.0 * synth.uniform01(3, 0, 200000) - 1.0
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-8 + 2**-20], np.float32)
    got = synth.to_bf16_bits(vals)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa wins (1.0); 1+3*2^-8 rounds up to 1+2^-6
    assert list(got) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]
    assert np.array_equal(synth.bf16_bits_to_fp32(got)[[0, 3]], np.array([1.0, -2.5], np.float32))


def test_oracle_rejects_bad_arguments():
    Q = np.zeros((1, 1, 2, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.attn_fwd(Q, np.zeros((1, 1, 0, 2), np.float32), np.zeros((1, 1, 0, 2), np.float32), 1.0, False)
    with pytest.raises(ValueError):
        oracle.attn_rows(Q, Q, Q, 1.0, False, [[0, 0, 5]])


# ---- mutation check: each planted mistake must fail an independent pin -------------------------

MUTANTS = {
    "score_sign_flipped": ("s[n] = J->scale * dot;", "s[n] = -J->scale * dot;"),
    "causal_off_by_one": ("case ORC_MASK_CAUSAL: return j <= i + J->offset;",
                          "case ORC_MASK_CAUSAL: return j <= i + J->offset + 1;"),
    "max_shift_dropped": ("exp(s[n] - m)", "exp(s[n])"),
    "scale_ignored": ("s[n] = J->scale * dot;", "s[n] = dot;"),
    "dot_term_dropped": ("for (int64_t d = 0; d < J->D_qk; ++d)\n            dot +=",
                         "for (int64_t d = 1; d < J->D_qk; ++d)\n            dot +="),
    "value_rows_reversed": ("const int64_t v0 = (kv * J->S_k + keys[n]) * J->D_v;",
                            "const int64_t v0 = (kv * J->S_k + keys[n_keys - 1 - n]) * J->D_v;"),
    "key_head_ignored": ("const int64_t k0 = (kv * J->S_k + j) * J->D_qk;",
                         "const int64_t k0 = ((b * J->H_kv) * J->S_k + j) * J->D_qk;"),
    "normalisation_dropped": ("const double w = exp(s[n] - m) / l;", "const double w = exp(s[n] - m);"),
    "query_row_fixed": ("const int64_t q0 = ((b * J->H + h) * J->S_q + i) * J->D_qk;",
                        "const int64_t q0 = ((b * J->H + h) * J->S_q + 0) * J->D_qk;"),
    "bf16_widening_shift": ("<< 16", "<< 15"),
    # grouped heads, offsets, windows and the log-sum-exp
    "kv_head_modulo": ("const int64_t g = h / (J->H / J->H_kv);", "const int64_t g = h % J->H_kv;"),
    "offset_ignored": ("case ORC_MASK_CAUSAL: return j <= i + J->offset;", "case ORC_MASK_CAUSAL: return j <= i;"),
    "offset_sign_flipped": ("case ORC_MASK_CAUSAL: return j <= i + J->offset;",
                            "case ORC_MASK_CAUSAL: return j + J->offset <= i;"),
    "window_too_wide": ("return i + J->offset - J->window < j && j <= i + J->offset;",
                        "return i + J->offset - J->window <= j && j <= i + J->offset;"),
    "window_without_offset": ("return i + J->offset - J->window < j && j <= i + J->offset;",
                              "return i - J->window < j && j <= i;"),
    "complement_off_by_one": ("case ORC_MASK_WINDOW_COMPLEMENT: return j <= i + J->offset - J->window;",
                              "case ORC_MASK_WINDOW_COMPLEMENT: return j < i + J->offset - J->window;"),
    "lse_max_dropped": ("*lse = n_keys > 0 ? m + log(l) : -INFINITY;", "*lse = n_keys > 0 ? log(l) : -INFINITY;"),
    "lse_base2": ("*lse = n_keys > 0 ? m + log(l) : -INFINITY;", "*lse = n_keys > 0 ? m + log2(l) : -INFINITY;"),
    "empty_row_lse_zero": ("*lse = n_keys > 0 ? m + log(l) : -INFINITY;", "*lse = n_keys > 0 ? m + log(l) : 0.0;"),
    "noop_control": ("case ORC_MASK_CAUSAL: return j <= i + J->offset;\n",
                     "case ORC_MASK_CAUSAL: return j <= i + J->offset + 0;\n"),
}
# "noop_control" changes nothing; it is checked to pass every pin (the harness itself is sound).
CONTROL = "noop_control"


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, mutant_dir):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutation site for {name} not found"
    msrc = os.path.join(mutant_dir, f"{name}.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load(oracle.build(msrc, os.path.join(mutant_dir, f"lib{name}.so")))
    failed = []
    for pin in pins.INDEPENDENT_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    if name == CONTROL:
        assert failed == [], f"control mutant should pass every pin, failed {failed}"
    else:
        assert failed, f"no independent pin caught the planted mistake {name}"
