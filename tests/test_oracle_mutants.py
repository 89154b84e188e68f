"""The oracle's pins catch the mistakes an oracle could plausibly hold.

Each case copies the C++ oracle's sources, plants one mistake in the copy (a text replacement of
one expression), builds the copy with the same compiler command, swaps it in for the real oracle
and runs the pins that should catch that mistake: at least one of them must fail.  The mistakes are
the readings the pages leave room for, or slips in writing them out:
eps outside the root ("Llama Architecture ...", Mathematical Foundations 1 prints it so), pairs
split by halves instead of interleaved, the rotation's sign, the head map h mod n_kv instead of
floor(h / r), no causal mask, no 1/sqrt(hd) scale, a dropped residual, gate and up swapped, E4M3
ties away from even, and sampling ties to the higher id.  Nothing here runs on a GPU.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

import pytest

from oracle import _lib
from tests import test_oracle_block_library as LIB
from tests import test_oracle_fp8_pins as F8
from tests import test_oracle_pins as P
from tests import test_oracle_sampling_pins as SP

# (name, file, original text, planted text, pins that must catch it)
MUTANTS = [
    ("eps outside the root", "llama_oracle.cpp", "std::sqrt(ss / (double)d + eps)", "(std::sqrt(ss / (double)d) + eps)",
     [P.test_rmsnorm_eps_inside_sqrt]),
    ("half-split RoPE pairs", "llama_oracle.cpp", "const double x0 = xp[2 * k], x1 = xp[2 * k + 1];",
     "const double x0 = xp[k], x1 = xp[k + hd / 2];",
     [P.test_rope_interleaved_pairs_and_theta_uses_head_dim,
      lambda: LIB.test_block_prefill_matches_library_formulation(4, 2)]),
    ("rotation by -m theta", "llama_oracle.cpp", "s = std::sin(ang);", "s = -std::sin(ang);",
     [P.test_rope_hd2_is_rotation_by_m]),
    ("head map h mod n_kv", "llama_oracle.cpp", "return h / (n_q / n_kv);", "return h % n_kv;",
     [P.test_toy_head_map, P.test_toy_outputs_match_page_and_closed_form]),
    ("no causal mask", "llama_oracle.cpp", "return n < (double)Tk ? (int64_t)n : Tk;", "return Tk;",
     [P.test_causal_mask_brute_force_and_future_independence]),
    ("no softmax scale", "llama_oracle.cpp", "const double scale = 1.0 / std::sqrt((double)hd);",
     "const double scale = 1.0;", [P.test_toy_softmax_rows_match_page]),
    ("dropped FFN residual", "llama_oracle.cpp", "y[i] = h[(size_t)i] + f[(size_t)i];", "y[i] = f[(size_t)i];",
     [P.test_block_identity_when_sublayers_output_zero]),
    ("gate and up swapped", "llama_oracle.cpp", "oracle_silu(gate.data(), rows * d_ff, m.data());",
     "oracle_silu(up.data(), rows * d_ff, m.data()); std::swap(gate, up);", [P.test_swiglu_gate_and_up_roles]),
    ("E4M3 ties away from even", "e4m3.cpp", "(d_hi == d_lo && (hi & 1) == 0)", "(d_hi == d_lo)",
     [F8.test_round_to_nearest_even_and_saturation]),
    ("ties to the higher id", "sampling.cpp", "std::iota(ids.begin(), ids.end(), 0);",
     "std::iota(ids.begin(), ids.end(), 0); std::reverse(ids.begin(), ids.end());",
     [SP.test_argmax_and_ties_to_lower_id]),
]


@pytest.fixture(scope="module")
def mutant_builds(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not found")
    root = tmp_path_factory.mktemp("oracle_mutants")

    def build(i):
        name, fname, old, new, _ = MUTANTS[i]
        d = root / f"m{i}"
        d.mkdir()
        for f in _lib.SOURCES + [_lib.HEADER]:
            shutil.copy(os.path.join(_lib.DIR, f), d / f)
        text = (d / fname).read_text()
        assert text.count(old) == 1, f"{name}: the expression to replace is not in {fname} exactly once"
        (d / fname).write_text(text.replace(old, new))
        so = str(d / "liboracle_mutant.so")
        subprocess.check_call(_lib.build_cmd(so, src_dir=str(d)))
        return so

    with cf.ThreadPoolExecutor(max_workers=4) as ex:
        return list(ex.map(build, range(len(MUTANTS))))


@pytest.mark.parametrize("i", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(i, mutant_builds):
    name, _, _, _, pins = MUTANTS[i]
    real = _lib.lib()
    caught = []
    try:
        _lib._lib = _lib.load(mutant_builds[i])
        for pin in pins:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    finally:
        _lib._lib = real
    assert caught, f"no pin caught the planted mistake '{name}'"


def test_the_real_oracle_passes_the_same_pins():
    for *_, pins in MUTANTS:
        for pin in pins:
            pin()
