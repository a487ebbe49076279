"""Mutation tests for the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source --
a wrong head mapping, an off-by-one in the causal limit, a dropped term, a
transposed operand -- builds the copy with gcc into a temporary directory and
runs the pins against it. At least one pin must fail for every mutant,
otherwise the pins would not have caught that mistake in the real oracle.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    # interleaved instead of contiguous groups
    "mapping_mod": ("const int g = h / heads_per_group;", "const int g = h % G;"),
    # off-by-one in the last visible key
    "causal_off_by_one": ("const long last = (long)T - sq + s;",
                          "const long last = (long)T - sq + s - 1;"),
    # no mask among the new tokens (every row sees the whole cache)
    "causal_dropped": ("const long last = (long)T - sq + s;", "const long last = (long)T - 1;"),
    # top-left aligned mask
    "causal_top_left": ("const long last = (long)T - sq + s;", "const long last = (long)s;"),
    # lse without the max term
    "lse_drops_mu": ("lse[r] = mu + log(Z);", "lse[r] = log(Z);"),
    # output not normalised by the softmax denominator
    "no_normalise": ("orow[d] /= Z;", "orow[d] /= 1.0;"),
    # scale not applied
    "scale_dropped": ("x[t] = scale * dot;", "x[t] = dot;"),
    # q read as [B, H, sq, D] (transposed operand)
    "q_transposed": ("const uint16_t* qrow = q + (((long)b * sq + s) * H + h) * D;",
                     "const uint16_t* qrow = q + (((long)b * H + h) * sq + s) * D;"),
    # V rows taken in reverse order
    "v_reversed": ("w * bf16_bits_to_double(vbase[t * D + d]);",
                   "w * bf16_bits_to_double(vbase[(n - 1 - t) * D + d]);"),
    # K read from the V cache
    "k_from_v": ("bf16_bits_to_double(kbase[t * D + d]);", "bf16_bits_to_double(vbase[t * D + d]);"),
    # wrong sign in the exponent
    "exp_sign": ("exp(x[t] - mu)", "exp(mu - x[t])"),
    # wrong row decomposition for s
    "row_decomp": ("const int s = (int)((r / H) % sq);", "const int s = (int)(r % sq);"),
    # empty rows produce garbage instead of out = 0, lse = -inf
    "empty_row_lse": ("lse[r] = -INFINITY;", "lse[r] = 0.0;"),
}


def _run_pins(orc):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        if pin.__name__ == "pin_bruteforce_mpmath":
            try:
                import mpmath  # noqa: F401
            except ImportError:
                continue
        try:
            pin(orc)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failed.append((pin.__name__, type(e).__name__))
    return failed


def test_every_mutation_target_exists():
    src = open(oracle.SOURCE).read()
    for name, (old, _new) in MUTANTS.items():
        assert old in src, name


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    mutated = src.replace(old, new)
    assert mutated != src
    path = os.path.join(tmp_path, f"mutant_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.compile_oracle(path, os.path.join(tmp_path, f"libmutant_{name}.so"))
    failed = _run_pins(oracle.Oracle(lib))
    assert failed, f"no pin catches mutant {name}"
