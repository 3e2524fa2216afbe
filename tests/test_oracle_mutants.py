"""The oracle's pins catch plausible mistakes. Each case plants one mistake
in a copy of oracle/fsdp_oracle.c (on the CPU), builds it, and runs the pin
suites against that build in a subprocess: they must fail. A mistake that
survives would mean the pins cannot tell it from the method."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fsdp_oracle.c")

# (name, exact text in the source, replacement)
MUTANTS = [
    ("sum_reverse_order",
     "for (int64_t q = 1; q < N; ++q) acc = acc + grad_at(G[q], grad_dtype, j);\n        g[i] = acc * c;",
     "for (int64_t q = N - 1; q >= 1; --q) acc = grad_at(G[q], grad_dtype, j) + acc;\n        g[i] = acc * c;"),
    ("no_average", "s->c = (float)(1.0 / ((double)world * (double)h->grad_scale));",
     "s->c = (float)(1.0 / (double)h->grad_scale);"),
    ("no_unscale", "s->c = (float)(1.0 / ((double)world * (double)h->grad_scale));",
     "s->c = (float)(1.0 / (double)world);"),
    ("decay_sign", "s->decay = (float)(1.0 - (double)h->lr * (double)h->weight_decay);",
     "s->decay = (float)(1.0 + (double)h->lr * (double)h->weight_decay);"),
    ("no_bias_correction_m", "s->alpha = (float)((double)h->lr / (1.0 - pow((double)h->beta1, t)));",
     "s->alpha = h->lr;"),
    ("no_bias_correction_v", "s->b2s = (float)sqrt(1.0 - pow((double)h->beta2, t));", "s->b2s = 1.0f;"),
    ("bias_correction_off_by_one", "s->alpha = (float)((double)h->lr / (1.0 - pow((double)h->beta1, t)));",
     "s->alpha = (float)((double)h->lr / (1.0 - pow((double)h->beta1, t + 1.0)));"),
    ("eps_inside_sqrt", "float denom = sqrtf(vi) / s->b2s + s->eps;\n        pi = pi - s->alpha * (mi / denom);\n        p[i] = pi;",
     "float denom = sqrtf(vi + s->eps) / s->b2s;\n        pi = pi - s->alpha * (mi / denom);\n        p[i] = pi;"),
    ("betas_swapped", "float mi = s->beta1 * m[i] + s->one_minus_beta1 * gi;",
     "float mi = s->beta2 * m[i] + s->one_minus_beta2 * gi;"),
    ("v_without_square", "float vi = s->beta2 * v[i] + s->one_minus_beta2 * (gi * gi);",
     "float vi = s->beta2 * v[i] + s->one_minus_beta2 * fabsf(gi);"),
    ("update_sign", "pi = pi - s->alpha * (mi / denom);\n        p[i] = pi;",
     "pi = pi + s->alpha * (mi / denom);\n        p[i] = pi;"),
    ("decay_after_update", "float pi = p[i] * s->decay;\n        float mi",
     "float pi = p[i];\n        float mi"),
    ("bf16_truncates", "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;\n    return (uint16_t)kept;",
     "return (uint16_t)kept;"),
    ("bf16_ties_away", "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;",
     "if (dropped >= 0x8000u) kept += 1u;"),
    ("f16_ties_away", "if (dropped > 0x1000u || (dropped == 0x1000u && (kept & 1u))) h += 1u;",
     "if (dropped >= 0x1000u) h += 1u;"),
    ("shard_interleaved", "int64_t j = rank * S + i;\n        float acc = grad_at(G[0], grad_dtype, j);\n        for (int64_t q = 1; q < N; ++q) acc = acc + grad_at",
     "int64_t j = i * N + rank;\n        float acc = grad_at(G[0], grad_dtype, j);\n        for (int64_t q = 1; q < N; ++q) acc = acc + grad_at"),
    ("pad_at_front", "unsigned char *out = (unsigned char *)dst;\n    int64_t at = 0;\n    for (int k = 0; k < n; ++k) {\n        memcpy",
     "unsigned char *out = (unsigned char *)dst;\n    int64_t at = padded;\n    for (int k = 0; k < n; ++k) at -= numels[k];\n"
     "    memset(out, 0, (size_t)(at * elem_size));\n    for (int k = 0; k < n; ++k) {\n        memcpy"),
    ("gather_reversed", "memcpy(out + (size_t)(r * S) * elem_size, shards[r], (size_t)S * elem_size);",
     "memcpy(out + (size_t)((N - 1 - r) * S) * elem_size, shards[r], (size_t)S * elem_size);"),
    ("sgd_dampened", "float b = h->step == 1 ? d : h->beta1 * *s0 + d;",
     "float b = h->step == 1 ? d : h->beta1 * *s0 + (1.0f - h->beta1) * d;"),
    ("sgd_no_weight_decay", "float d = g + h->weight_decay * pi;\n        float b =",
     "float d = g;\n        float b ="),
    ("adamax_min", "float ui = (a > b || a != a) ? a : b;", "float ui = (a < b || a != a) ? a : b;"),
    ("adamax_no_eps", "float a = s->beta2 * *s1, b = fabsf(d) + s->eps;", "float a = s->beta2 * *s1, b = fabsf(d);"),
    ("adadelta_ratio_inverted", "float delta = (sqrtf(*s1 + s->eps) / sqrtf(sq + s->eps)) * d;",
     "float delta = (sqrtf(sq + s->eps) / sqrtf(*s1 + s->eps)) * d;"),
    ("adadelta_stale_square", "float delta = (sqrtf(*s1 + s->eps) / sqrtf(sq + s->eps)) * d;",
     "float delta = (sqrtf(*s1 + s->eps) / sqrtf(*s0 + s->eps)) * d;"),
    ("lowp_reduce_not_rounded", "for (int64_t q = 1; q < N; ++q) acc = round_to(grad_dtype, acc + grad_at(G[q], grad_dtype, j));",
     "for (int64_t q = 1; q < N; ++q) acc = acc + grad_at(G[q], grad_dtype, j);"),
    ("lowp_state_truncates", "((uint16_t *)base)[j] = orc_f32_to_bf16(x);",
     "((uint16_t *)base)[j] = (uint16_t)(f32_bits(x) >> 16);"),
    ("shadow_no_unscale", "G_avg[j] = acc / ((double)N * grad_scale);", "G_avg[j] = acc / (double)N;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    import oracle
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {name}"
    mutant = tmp_path / f"{name}.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant), str(tmp_path / f"lib{name}.so"))
    env = dict(os.environ, FSDP_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_pins_next.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not catch the planted mistake {name}"
