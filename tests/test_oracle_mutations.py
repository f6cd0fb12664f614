"""The pins are strong enough: plant one plausible mistake at a time in a copy of
the oracle's C source (on the CPU, in a temporary directory), rebuild it, and
check that at least one pin from test_oracle_pins.py fails against it."""
import importlib.util
import os
import shutil

import pytest

import tests.test_oracle_fp8 as fp8_pins
import tests.test_oracle_pins as pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("score_sign", "s[i] = J->scale * dot;", "s[i] = -J->scale * dot;"),
    ("scale_dropped", "s[i] = J->scale * dot;", "s[i] = dot;"),
    ("lse_without_max", "if (lse) *lse = M + log(sum);", "if (lse) *lse = log(sum);"),
    ("k_v_swapped", "cache_row(pb, 0, g, (int)(i % J->bs)", "cache_row(pb, 1, g, (int)(i % J->bs)"),
    ("gqa_modulo", "int g = h / group;", "int g = h % J->hkv;"),
    ("causal_off_by_one", "(long)L - q_len + r + 1", "(long)L - q_len + r"),
    ("causal_top_left", "(long)L - q_len + r + 1", "r + 1"),
    ("offset_xor", "size_t kr = cache_row(pb, 0, g, (int)(i % J->bs)",
     "size_t kr = cache_row(pb, 0, g, (int)((i % J->bs) ^ 1)"),
    ("last_key_dropped", "for (long i = 0; i < kmax; ++i) {\n        double w", "for (long i = 0; i + 1 < kmax; ++i) {\n        double w"),
    ("combine_weight_inverted", "double w = exp(ls[s] - M);", "double w = exp(M - ls[s]);"),
    ("append_ignores_ctx_before", "long pos = (long)ctx_before[b] + (t - cu_new_lens[b]);",
     "long pos = (t - cu_new_lens[b]);"),
    ("layout_kv_inner", "return ((((size_t)pb * 2 + kv) * hkv + h) * bs + off) * (size_t)d;",
     "return ((((size_t)pb * hkv + h) * 2 + kv) * bs + off) * (size_t)d;"),
    ("half_exponent_bias", "v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
    ("bf16_shift", "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
]

PIN_TESTS = [
    ("test_append_contiguous_special_case", {}),
    ("test_append_in_two_steps_equals_one", {}),
    ("test_decode_matches_library_sdpa", dict(dtype="f16", hq=8, hkv=2)),
    ("test_decode_matches_library_sdpa", dict(dtype="bf16", hq=4, hkv=4)),
    ("test_causal_prefill_matches_library_sdpa", dict(q_lens=(7, 3), lens=(50, 3))),
    ("test_lse_matches_logsumexp", {}),
    ("test_combine_of_splits_equals_unsplit", dict(bounds=[(0, 64), (64, 200)])),
]


def load_mutant(tmp_path, name, old, new):
    d = tmp_path / ("oracle_" + name)
    shutil.copytree(ORACLE_DIR, d, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    src = (d / "oracle.c").read_text()
    assert src.count(old) == 1, name
    (d / "oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle_mut_" + name, str(d / "__init__.py"),
                                                  submodule_search_locations=[str(d)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_some_pin_fails_on_planted_mistake(tmp_path, monkeypatch, name, old, new):
    mutant = load_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(pins, "oracle", mutant)
    failed = []
    for fn, kw in PIN_TESTS:
        try:
            getattr(pins, fn)(**kw)
        except (AssertionError, ValueError):
            failed.append(fn)
    assert failed, "no pin caught mutation %s" % name


# The FP8 cache: the E4M3 conversion, the quantising append and the dequantising attention.
FP8_MUTATIONS = [
    ("e4m3_exponent_bias", "else v = ldexp((double)(8 + m), e - 10);", "else v = ldexp((double)(8 + m), e - 9);"),
    ("e4m3_rounds_up", "double r = rint(ldexp(a, 3 - e)) - 8.0;", "double r = ceil(ldexp(a, 3 - e)) - 8.0;"),
    ("e4m3_ties_away", "double r = rint(ldexp(a, 3 - e)) - 8.0;", "double r = round(ldexp(a, 3 - e)) - 8.0;"),
    ("e4m3_subnormal_step", "double q = rint(a * 512.0);", "double q = rint(a * 256.0);"),
    ("fp8_scale_inverted", "float scale = amax / 448.0f;", "float scale = 448.0f / amax;"),
    ("fp8_codes_unscaled", "float y = (float)to_double(dtype, src[e]) * inv;",
     "float y = (float)to_double(dtype, src[e]);"),
    ("fp8_first_scale_only", "* (double)J->scales[row / (size_t)J->d];", "* (double)J->scales[0];"),
    ("fp8_scale_dropped", "* (double)J->scales[row / (size_t)J->d];", ";"),
]

FP8_PIN_TESTS = [
    ("test_decode_every_code_matches_torch", {}),
    ("test_encode_matches_torch_in_range_including_ties", {}),
    ("test_encode_ties_go_to_even_and_saturates", {}),
    ("test_append_follows_the_definition", {}),
    ("test_append_roundtrip_error_bound", {}),
    ("test_attention_over_fp8_is_softmax_of_dequantised", dict(causal=False, q_lens=None)),
]


@pytest.mark.parametrize("name,old,new", FP8_MUTATIONS, ids=[m[0] for m in FP8_MUTATIONS])
def test_some_fp8_pin_fails_on_planted_mistake(tmp_path, monkeypatch, name, old, new):
    mutant = load_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(fp8_pins, "oracle", mutant)
    failed = []
    for fn, kw in FP8_PIN_TESTS:
        try:
            getattr(fp8_pins, fn)(**kw)
        except (AssertionError, ValueError):
            failed.append(fn)
    assert failed, "no pin caught mutation %s" % name
