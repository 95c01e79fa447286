"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source
(never in the oracle itself), builds it, and runs the oracle pin tests against
that build; they must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")
PIN_TESTS = ["tests/test_oracle_step.py", "tests/test_oracle_formats.py",
             "tests/test_oracle_quant.py", "tests/test_oracle_ckpt.py",
             "tests/test_oracle_offload.py"]

MUTANTS = {
    "reduce-reverse-rank-order": ("for (int r = 0; r < nd; r++)\n            s = s +",
                                  "for (int r = nd - 1; r >= 0; r--)\n            s = s +"),
    "reduce-transposed-index": ("grads[(int64_t)r * rank_stride + i]", "grads[i * nd + r]"),
    "reduce-no-average": ("float avg = s / (float)nd;", "float avg = s;"),
    "reduce-no-unscale": ("float gi  = avg / loss_scale;", "float gi  = avg;"),
    "adam-no-bias-correction-m": ("float mhat = mi / bc1;", "float mhat = mi;"),
    "adam-eps-inside-sqrt": ("(sqrtf(vhat) + hp->eps)", "sqrtf(vhat + hp->eps)"),
    "adam-v-of-g-not-g2": ("omb2 * (gi * gi)", "omb2 * gi"),
    "adam-betas-swapped-in-m": ("hp->beta1 * m[i] + omb1 * gi", "hp->beta2 * m[i] + omb2 * gi"),
    "adam-wrong-sign": ("p = p - hp->lr * upd;", "p = p + hp->lr * upd;"),
    "adamw-decay-dropped": ("if (hp->decoupled_wd) p  = p * decay;",
                            "if (hp->decoupled_wd) p  = p;"),
    "bias-correction-stuck-at-t1": ("st->beta1_pow = st->beta1_pow * (double)hp->beta1;",
                                    "st->beta1_pow = (double)hp->beta1;"),
    "clip-always": ("if (clip > 0.0f && norm > (double)clip)", "if (clip > 0.0f)"),
    "norm-squares-in-float": ("acc = acc + (double)g[i] * (double)g[i];",
                              "acc = acc + (double)(g[i] * g[i]);"),
    "skip-keeps-scale": ("st->loss_scale = st->loss_scale * hp->backoff;",
                         "st->loss_scale = st->loss_scale;"),
    "skip-advances-t": ("res->skipped  = 1;", "res->skipped  = 1; st->t = st->t + 1;"),
    "static-skip-ignored": ("if (overflow && (hp->dynamic_scale || hp->skip_on_overflow)) {",
                            "if (overflow && hp->dynamic_scale) {"),
    "static-skip-backs-off": ("        if (hp->dynamic_scale) {\n            st->loss_scale",
                              "        {\n            st->loss_scale"),
    "round-ties-away": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;\n    return r * q;",
                        "if (frac > 0.5 || (frac == 0.5)) r += 1.0;\n    return r * q;"),
    "qwz-round-ties-away": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;\n    return (int32_t)r;",
                            "if (frac > 0.5 || (frac == 0.5)) r += 1.0;\n    return (int32_t)r;"),
    "gather-off-by-one": ("out[j] = slices[k][j % slice];",
                          "out[j] = slices[k][(j + 1) % slice];"),
    "qwz-qmax-off-by-one": ("const float qmax = (float)((1 << (bits - 1)) - 1);",
                            "const float qmax = (float)(1 << (bits - 1));"),
    "qwz-nibble-order": ("if (i % 2 == 0) q[i / 2] = (uint8_t)((q[i / 2] & 0xF0) | nib);",
                         "if (i % 2 == 1) q[i / 2] = (uint8_t)((q[i / 2] & 0xF0) | nib);"),
    "qwz-truncate": ("code = round_half_even_to_int(x[i] / scale);",
                     "code = (int32_t)(x[i] / scale);"),
    "qwz-gather-ignores-offset": ("int64_t e = offset + j % slice;", "int64_t e = j % slice;"),
    "reshard-padding-kept": ("else memset(dst, 0, (size_t)elem_bytes);", "else { }"),
    "layout-slice-start-dropped": ("int64_t local = (int64_t)r * s + (j - slice_start);",
                                   "int64_t local = (int64_t)r * s + j;"),
    "layout-unit-start-dropped": ("return local < L->len[u] ? unit_start + local : -1;",
                                  "return local < L->len[u] ? local : -1;"),
    "layout-boundary-off-by-one": ("if (j < slice_start + s) {", "if (j <= slice_start + s) {"),
    "reshard-ranks-reversed": ("int64_t g = zo_layout_global(A, r, j);",
                               "int64_t g = zo_layout_global(A, A->nd - 1 - r, j);"),
    "offload-no-rounding": ("float gi = to_float(dtype, q) / loss_scale;",
                            "float gi = mean / loss_scale;"),
    "offload-unscale-before-round": ("uint16_t q = from_float(dtype, mean);",
                                     "uint16_t q = from_float(dtype, mean / loss_scale);"),
    "offload-no-average": ("float mean = sum / (float)nd;", "float mean = sum;"),
    "offload-clip-dropped": ("res->clip_coef = zo_clip_coef(res->grad_norm, hp->clip_norm);\n"
                             "    zo_advance(hp, st, bad, res);",
                             "res->clip_coef = 1.0f;\n    zo_advance(hp, st, bad, res);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "zero_oracle.c"
    mut.write_text(src.replace(old, new))
    (tmp_path / "zero_oracle.h").write_text(open(SRC[:-1] + "h").read())
    so = tmp_path / "libmutant.so"
    sys.path.insert(0, ROOT)
    import oracle
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(mut), "-lm"], check=True)
    env = dict(os.environ, ZO_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
