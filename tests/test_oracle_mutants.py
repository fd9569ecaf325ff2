"""The oracle's pins have teeth: plant a plausible mistake in a copy of the
oracle's C source (on the CPU), rebuild it, and check that at least one pin
fails on it.  The committed oracle itself is untouched."""
import os
import subprocess

import pytest

import oracle
import test_oracle_attention as A
import test_oracle_codecs as Cd

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("scale dropped", "s[t] = scale * acc;", "s[t] = acc;"),
    ("gqa head mapping", "(int32_t)(h / group),\n                                qd, seq_lens[b]",
     "(int32_t)(h % num_kv_heads),\n                                qd, seq_lens[b]"),
    ("causal mask off by one", "nkeys = last + 1 < lk ? last + 1 : lk;", "nkeys = last < lk ? last : lk;"),
    ("max subtraction sign", "s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    ("cache layout transposed", "((blk * num_kv_heads + h) * block_size + off) * head_size + d",
     "((blk * block_size + off) * num_kv_heads + h) * head_size + d"),
    ("token offset in page", "int64_t blk = table_row[t / bs], off = t % bs;\n        double acc",
     "int64_t blk = table_row[t / bs], off = (t + 1) % bs;\n        double acc"),
    ("decode length off by one", "qd, seq_lens[b], scale, o, s);", "qd, seq_lens[b] - 1, scale, o, s);"),
    ("softmax not normalised", "double p = s[t] / l;", "double p = s[t];"),
    ("rounding ties away", "nearbyint(x / ulp)", "round(x / ulp)"),
    ("fp8 multiply instead of divide", "volatile float qk = xk / k_scale;", "volatile float qk = xk * k_scale;"),
    ("fp8 no saturation", "if (fabs(r) > 448.0) r = signbit(r) ? -448.0 : 448.0;", ""),
    ("bf16 exponent bias", "decode_fields(b, 7, -126, 127, 8)", "decode_fields(b, 7, -126, 126, 8)"),
    ("value row from key cache", "double vd = load_elem(c->v_cache", "double vd = load_elem(c->k_cache"),
]

PINS = [
    lambda: [A.test_decode_matches_sdpa(c) for c in A.CASES],
    A.test_closed_form_single_key_returns_v_row,
    A.test_gqa_head_mapping_is_contiguous_groups,
    A.test_p2_decode_example_slots_and_attention,
    A.test_unreferenced_and_masked_slots_do_not_matter,
    lambda: A.test_prefill_matches_sdpa(True),
    A.test_p2_varlen_example,
    lambda: A.test_cache_write_e4m3_quantizes_x_over_scale(1),
    Cd.test_bf16_decode_all_codes,
    Cd.test_e4m3_encode_satfinite,
    Cd.test_f16_encode_from_double,
]


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    src = open(SRC).read()
    d = tmp_path_factory.mktemp("mutants")
    libs = {}
    for i, (name, old, new) in enumerate(MUTANTS):
        assert src.count(old) == 1, name
        path = d / f"m{i}.c"
        path.write_text(src.replace(old, new))
        so = d / f"m{i}.so"
        subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"],
                       check=True)
        libs[name] = str(so)
    return libs


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(mutant_libs, name):
    prev = oracle.use_library(mutant_libs[name])
    caught = []
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin)
                break
    finally:
        oracle.restore_library(prev)
    assert caught, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_all_pins():
    oracle.lib()
    for pin in PINS:
        pin()
