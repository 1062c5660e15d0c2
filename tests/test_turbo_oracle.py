"""The TurboAdam-style oracle against its pins (CPU only), and planted mistakes
in copies of turbo.c that the pins must catch."""
import os

import numpy as np
import pytest

import oracle
import pins_turbo

with open(oracle.TURBO_SOURCE) as _f:
    _SRC = _f.read()


@pytest.mark.parametrize("name", sorted(pins_turbo.ALL_CHECKS))
def test_turbo_oracle_pin(name):
    pins_turbo.ALL_CHECKS[name](oracle.default())


MUTANTS = [
    ("grid_intervals_off_by_one", "return float_of((uint32_t)(blo + num / (uint64_t)(K - 1)));",
     "return float_of((uint32_t)(blo + num / (uint64_t)K));", ["q1_grid_closed_forms"]),
    ("upper_endpoint_not_rounded_up", "*hi = (mx == ldexpf(1.0f, e)) ? e : e + 1;", "*hi = e;",
     ["q1_endpoints"]),
    ("rounds_up_on_large_u", "return (u < p) ? j + 1 : j;", "return (u > p) ? j + 1 : j;",
     ["q1_rounding"]),
    ("ustate_rounds_up_on_large_u", "return (u < frac) ? j + 1 : j;",
     "return (u > frac) ? j + 1 : j;", ["ustate_code"]),
    ("no_recentring", "float delta = (sdec * (float)S) / (float)(2 * c);", "float delta = 0.0f;",
     ["means_recentred", "first_moment_reconstructed"]),
    ("q_normalised_by_exact_v", "float den = sqrtf(vhat[k + j] / h.bc2) + h.ef;",
     "float den = sqrtf(vnew[k + j] / h.bc2) + h.ef;",
     ["means_recentred"]),
    ("scales_not_rotated", "uscal[0] = uscal[1];", "uscal[0] = uscal[0];",
     ["finalize_rotates_scales"]),
    ("prior_first_moment_not_rescaled", "m = (q * den) * bc1p;", "m = q * bc1p;",
     ["step_is_adamw_on_decoded_moments", "first_moment_reconstructed"]),
    ("mean_not_divided", "float mean = tree_sum64(qv) / (float)c;", "float mean = tree_sum64(qv);",
     ["means_recentred"]),
    ("hash_counter_not_advanced", "return oracle_splitmix64_mix(seed + (counter + 1u) * 0x9E3779B97F4A7C15ull);",
     "return oracle_splitmix64_mix(seed + counter);", ["counter_is_a_splitmix_position"]),
    ("odd_index_repeats_the_even_uniform", "uint64_t field = (index & 1u) ? (h >> 16) & 0xFFFFFFu : h >> 40;",
     "uint64_t field = h >> 40;", ["two_uniforms_per_output", "uniform_statistics"]),
    ("pair_counter_not_halved", "((uint64_t)stream << 40) | (index >> 1);",
     "((uint64_t)stream << 40) | index;", ["two_uniforms_per_output"]),
]


@pytest.mark.parametrize("name,old,new,expect", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_turbo_pins_catch_planted_mistake(name, old, new, expect, tmp_path):
    assert _SRC.count(old) == 1, f"mutation anchor not found once: {old!r}"
    src = tmp_path / f"{name}.c"
    src.write_text(_SRC.replace(old, new, 1))
    lib = oracle.compile_source(oracle.SOURCE, str(tmp_path / f"{name}.so"), turbo=str(src))
    orc = oracle.Oracle(os.path.abspath(lib))
    caught = []
    for pin in expect:
        try:
            pins_turbo.ALL_CHECKS[pin](orc)
        except AssertionError:
            caught.append(pin)
    assert caught, f"planted mistake {name} passed every pin in {expect}"


def test_turbo_slice_steps_as_in_the_whole_tensor():
    """Whole 128-value blocks are independent given the tensor's scales: the
    oracle's step over a slice (its rounding counters at the tensor's element
    indices) gives the slice of the whole-tensor step, p and every state
    array; only the RMS accumulator gathers the slice's squares alone."""
    n = 128 * 40 + 45
    rng = np.random.default_rng(21)
    orc = oracle.Oracle()
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = oracle.turbo_zero_state(n)
    for t in (1, 2, 3):
        g = (rng.normal(0, 1e-3, n) * rng.choice([1.0, 10.0], n)).astype(np.float32)
        p_next, st_next, _ = orc.turbo_step(p, g, st, t)
        for s0, length in ((0, 1024), (128 * 7, 128 * 5), (128 * 39, n - 128 * 39)):
            sl = {"ucode": st["ucode"][s0 // 4:(s0 + length + 3) // 4],
                  "umean": st["umean"][s0 // 64:(s0 + length + 63) // 64],
                  "uscal": st["uscal"].copy(),
                  "vidx": st["vidx"][s0 // 2:(s0 + length + 1) // 2],
                  "vend": st["vend"][2 * (s0 // 128):2 * ((s0 + length + 127) // 128)]}
            ps, sts, _ = orc.turbo_step(p[s0:s0 + length], g[s0:s0 + length], sl, t, index0=s0)
            assert np.array_equal(ps.view(np.uint32), p_next[s0:s0 + length].view(np.uint32))
            for k in ("ucode", "umean", "vidx", "vend"):
                whole = {"ucode": st_next["ucode"][s0 // 4:(s0 + length + 3) // 4],
                         "umean": st_next["umean"][s0 // 64:(s0 + length + 63) // 64],
                         "vidx": st_next["vidx"][s0 // 2:(s0 + length + 1) // 2],
                         "vend": st_next["vend"][2 * (s0 // 128):2 * ((s0 + length + 127) // 128)]}[k]
                assert np.array_equal(sts[k], whole), (t, s0, k)
        st_next["uscal"] = orc.turbo_finalize(st_next["uscal"], n, 1.1)
        p, st = p_next, st_next
