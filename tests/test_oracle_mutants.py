"""The pins can tell a wrong oracle from the right one: each case plants one
plausible mistake in a copy of the oracle's C++ source (an index off by one,
a dropped term, a flipped comparison or tie rule, a wrong normaliser),
builds it, loads it in place of the oracle and runs the pins that guard that
step; at least one of them must fail. No GPU involved."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "crisp_oracle.cpp")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MUTANTS = [
    ("slash block off by one", "s[(i - j) / kB] += m;", "s[(i - j + 1) / kB] += m;",
     [lambda: pins.test_vs_masses_single_entry_closed_form(10, 500),
      lambda: pins.test_vs_masses_single_entry_closed_form(127, 640)]),
    ("sink columns kept in the slash masses", "if (j <= i && j >= 128) s[", "if (j <= i && j >= 0) s[",
     [pins.test_vs_masses_sum_invariants, lambda: pins.test_vs_masses_single_entry_closed_form(5, 127)]),
    ("recency slice one column short", "if (j < sink || j >= n - recency) S += m;",
     "if (j < sink || j > n - recency) S += m;", [pins.test_cstruct_equals_brute_force_slice_sum]),
    ("slice union counted twice", "if (j < sink || j >= n - recency) S += m;",
     "if (j < sink) S += m;\n        if (j >= n - recency) S += m;",
     [lambda: pins.test_cstruct_other_slice_widths_brute_force(700, 500)]),
    ("route tie goes to PE", "route[h] = static_cast<unsigned __int128>(tau_den) * S >= ",
     "route[h] = static_cast<unsigned __int128>(tau_den) * S > ", [pins.test_route_tau_tie_goes_to_vs]),
    ("noise floor not strict", "if (lhs > rhs && !chosen[c])", "if (lhs >= rhs && !chosen[c])",
     [lambda: pins.test_select_vs_hand_fixture(GOLDEN), pins.test_select_vs_equal_masses_fill_lowest]),
    ("k_min fill ties by the higher index",
     "    if (m[a] != m[b]) return m[a] > m[b];\n    return a < b;\n  });\n  for (int c : rest)",
     "    if (m[a] != m[b]) return m[a] > m[b];\n    return a > b;\n  });\n  for (int c : rest)",
     [pins.test_select_vs_equal_masses_fill_lowest]),
    ("always-retained recency block dropped (coverage rule)", "if (dir == 0) chosen[nb - 1] = 1;",
     "if (dir == 0) chosen[nb - 2] = 1;", [pins.test_select_vs_gamma_sink_only_collapse,
                                          pins.test_select_vs_gamma_one_keeps_all_nonzero_and_zero_keeps_forced]),
    ("quanta truncated", "std::nearbyint(x)", "std::floor(x)", [pins.test_quantize_round_half_even]),
    ("attention without the 1/sqrt(d) scale", "s.push_back(scale * acc);", "s.push_back(acc);",
     [pins.test_dense_attention_matches_sdpa]),
    ("divergence in bits", "if (a > 0.0) kl_a += a * std::log(a / m);", "if (a > 0.0) kl_a += a * std::log2(a / m);",
     [pins.test_route_jsd_matches_scipy_jensenshannon]),
    ("slash band misses its second key block", "if (qb - s - 1 >= 0) set_bit(out, qb - s - 1);", "",
     [pins.test_build_mask_matches_token_level_definition]),
    ("short block pooled over 128 tokens",
     "dst[c] /= len;\n  });\n  parallel_for(static_cast<int64_t>(hkv) * nb",
     "dst[c] /= kB;\n  });\n  parallel_for(static_cast<int64_t>(hkv) * nb",
     [lambda: pins.test_ragged_pe_map_uses_block_means_over_own_tokens(300)]),
]


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_a_planted_mistake(tmp_path, monkeypatch, name, old, new, checks):
    src = open(SRC).read()
    assert src.count(old) == 1, "the mutation must name one place in the source"
    mutant = tmp_path / "mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(mutant), "-o", str(lib_path)])
    monkeypatch.setattr(oracle, "_lib", oracle._configure(ctypes.CDLL(str(lib_path))))
    caught = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin noticed: {name}"
