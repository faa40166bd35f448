"""Each plausible mistake planted in a copy of the oracle fails at least one pin (CPU only).

The mistakes are planted by text substitution in a temporary copy of the C source, which
is compiled with gcc into a temporary directory; the committed oracle is not touched."""
import os
import shutil

import pytest

import oracle as oracle_pkg
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "rimuru_oracle.c")

MUTANTS = {
    "gate_up_swapped": [("g[i] += x[r] * w1[", "g[i] += x[r] * w3["),
                        ("u[i] += x[r] * w3[", "u[i] += x[r] * w1[")],
    "silu_sign": [("g[i] / (1.0 + exp(-g[i]))", "g[i] / (1.0 + exp(g[i]))")],
    "tie_to_higher_index": [("return a < b;", "return a > b;")],
    "renorm_ignored": [("double denom = renorm ? sum_topk : sum_all;", "double denom = sum_all;")],
    "softmax_unshifted_numerator": [("double p = exp((double)l[order[j]] - m) / denom;",
                                     "double p = exp((double)l[order[j]]) / denom;")],
    "unstable_grouping": [("sorted[cursor[e]] = f;",
                           "sorted[offsets[e] + offsets[e + 1] - 1 - cursor[e]] = f;")],
    "w1_transposed": [("w1[(size_t)r * I + i]", "w1[(size_t)i * H + r]")],
    "w2_transposed": [("w2[(size_t)i * H + c]", "w2[(size_t)c * I + i]")],
    "combine_drops_last_slot": [("for (int j = 0; j < k; ++j) {\n        int f = t * k + j;\n        acc",
                                 "for (int j = 0; j < k - 1; ++j) {\n        int f = t * k + j;\n        acc")],
    "combine_unweighted": [("acc += wd[f] * yall", "acc += yall")],
    "bf16_fraction_scale": [("(double)frac / 128.0", "(double)frac / 256.0")],
    "bf16_byte_order": [("src[at] | ((uint16_t)src[at + 1] << 8)", "src[at + 1] | ((uint16_t)src[at] << 8)")],
    "token_index": [("int t = f / k;", "int t = f % k;")],
    "page_offset": [("uint64_t start = (uint64_t)page_id * page_bytes;",
                     "uint64_t start = (uint64_t)page_id * page_bytes + 2;")],
    "gate_bias_in_silu": [("h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(-u[i])) * u[i];")],
    "bf16_subnormal_scale": [("ldexp((double)frac, -126 - 7)", "ldexp((double)frac, -126 - 8)")],
    "bf16_exponent_bias": [("ldexp(1.0 + (double)frac / 128.0, expo - 127)",
                            "ldexp(1.0 + (double)frac / 128.0, expo - 126)")],
    "full_softmax_skips_expert0": [("for (int e = 0; e < E; ++e) sum_all +=",
                                    "for (int e = 1; e < E; ++e) sum_all +=")],
    "topk_ascending_values": [("if (l[a] > l[b]) return 1;\n  if (l[a] < l[b]) return 0;",
                               "if (l[a] < l[b]) return 1;\n  if (l[a] > l[b]) return 0;")],
}


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


def test_default_oracle_passes_every_pin():
    assert pins.failing_pins(oracle_pkg.Oracle()) == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, src_text, tmp_path):
    text = src_text
    for old, new in MUTANTS[name]:
        assert text.count(old) == 1, f"mutation site for {name} not found exactly once: {old!r}"
        text = text.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(text)
    lib = oracle_pkg.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    o = oracle_pkg.Oracle(oracle_pkg.load(lib))
    failed = pins.failing_pins(o)
    assert failed, f"mutant {name} passed every pin"
