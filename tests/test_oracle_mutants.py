"""Plant plausible mistakes in copies of the oracle (CPU only) and check that the pins catch
each one: a dropped term, a wrong sign, an off-by-one mask, a swapped operand, a missing
normalisation. The real oracle source is never modified; each mutant is a patched copy
compiled into a temporary directory."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "dropped_scale": ("s[j] = sm_scale * dot;", "s[j] = dot;"),
    "causal_off_by_one": ("if (causal && j > i + off)", "if (causal && j >= i + off)"),
    "causal_offset_sign": ("if (causal && j > i + off)", "if (causal && j > i - off)"),
    "causal_top_left": ("if (causal && j > i + off)", "if (causal && j > i)"),
    "kv_head_interleaved": ("int64_t kvh = b * J->Hkv + h / G;", "int64_t kvh = b * J->Hkv + h % J->Hkv;"),
    "kv_head_query_stride": ("int64_t kvh = b * J->Hkv + h / G;", "int64_t kvh = b * J->H + h / G;"),
    "length_clamp_to_nq": ("if (L > Nk) L = Nk;", "if (L > N) L = N;"),
    "padding_off_by_one": ("if (j >= L)", "if (j > L)"),
    "lse_dropped_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "no_normalisation": ("double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    "wrong_sign_exponent": ("double p = exp(s[j] - m) / l;", "double p = exp(m - s[j]) / l;"),
    "v_uses_k": ("o[c] += p * V[j * d + c];", "o[c] += p * K[j * d + c];"),
    "q_dot_v": ("dot += q[c] * K[j * d + c];", "dot += q[c] * V[j * d + c];"),
    "normaliser_without_mask": ("if (allowed(i, j, L, causal, off))\n            l += exp(s[j] - m);",
                                "if (1)\n            l += exp(s[j] - m);"),
    "decoder_bias": ("mag = ldexp((double)(1024 + f), e - 25);", "mag = ldexp((double)(1024 + f), e - 24);"),
    "subnormal_scale": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "bf16_exponent_bias": ("mag = ldexp((double)(128 + f), e - 134);",
                           "mag = ldexp((double)(128 + f), e - 133);"),
    "bf16_subnormal_scale": ("mag = ldexp((double)f, -133);", "mag = ldexp((double)f, -134);"),
    "bf16_read_as_f16": ("J.dec = dtype == 1 ? g_bf16_table : g_half_table;", "J.dec = g_half_table;"),
    "f32_read_as_16bit": ("if (J->dtype == 2) {", "if (J->dtype == 3) {"),
    "f32_wrong_stride": ("memcpy(&f, (const unsigned char *)base + idx * 4, sizeof f);",
                         "memcpy(&f, (const unsigned char *)base + idx * 2, sizeof f);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / f"mutant_{name}.c"
    mutated.write_text(src.replace(before, after))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / f"libmutant_{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception:  # an assertion, or an error the broken arithmetic provokes
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
