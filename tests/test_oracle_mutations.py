"""The pins bite: each plausible mistake planted in a copy of the oracle (on
the CPU) makes the pin suite fail.  The copy is compiled into a temporary
directory and loaded through ZERO_ORACLE_LIB in a child pytest process."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")

# (name, text in the oracle, planted replacement)
MUTANTS = [
    ("fold_reversed", "for (int32_t q = 1; q < n_ranks; ++q) acc = acc + orc_load_grad(grads[q], gdtype, i);",
     "for (int32_t q = n_ranks - 1; q >= 1; --q) acc = orc_load_grad(grads[q], gdtype, i) + acc;"),
    ("avg_by_reciprocal", "return acc / (float)n_ranks;", "return acc * (1.0f / (float)n_ranks);"),
    ("v_bracketing", "float vi = hp->b2 * v[i] + one_minus_b2 * g * g;",
     "float vi = hp->b2 * v[i] + one_minus_b2 * (g * g);"),
    ("bc2_without_sqrt", "*bc2 = sqrtf(1.0f - orc_powi(b2, t));", "*bc2 = 1.0f - orc_powi(b2, t);"),
    ("no_bias_correction_1", "*bc1 = 1.0f - orc_powi(b1, t);", "*bc1 = 1.0f;"),
    ("coupled_weight_decay", "float wi = w[i] * decay - lr_over_bc1 * mi / (sqrtf(vi) / bc2 + hp->eps);",
     "float wi = w[i] - lr_over_bc1 * (mi / (sqrtf(vi) / bc2 + hp->eps) + hp->wd * w[i]);"),
    ("eps_inside_sqrt", "(sqrtf(vi) / bc2 + hp->eps)", "(sqrtf(vi + hp->eps) / bc2)"),
    ("bf16_truncates", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;", "(void)lo;"),
    ("bf16_ties_away", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;", "if (lo >= 0x8000u) hi += 1u;"),
    ("pad_always", "return rem == 0 ? s : s + (quantum - rem);", "return s + (quantum - rem);"),
    ("pads_not_masked", "if (pad != NULL && pad[i]) return 0.0f;", ""),
    ("slice_stride", "map[(int64_t)r * H + hh + j] = f + (int64_t)r * hu + j;", "map[(int64_t)r * H + hh + j] = f + (int64_t)j * n_ranks + r;"),
    ("sqnorm_sum_in_float", "orc_sqacc_add_square(a, orc_avg_grad(n_ranks, grads, gdtype, pad, i));",
     "{ float q = orc_avg_grad(n_ranks, grads, gdtype, pad, i); orc_sqacc_add_square(a, sqrtf(q * q)); }"),
    ("clip_guard_dropped", "double c = (double)max_norm / (sqrt(S) + 1e-6);", "double c = (double)max_norm / sqrt(S);"),
    ("reshard_wrong_slice", "int64_t rs = k / h_from, js = k % h_from;", "int64_t rs = k / h_to, js = k % h_to;"),
    ("locate_wrong_rank", "rank[i] = (int32_t)(k / t[4 * u + 2]);", "rank[i] = (int32_t)(k % n_ranks);"),
    ("merge_drops_carry", "        dst->limb[k] = (uint64_t)t;\n        carry = (uint64_t)(t >> 64);",
     "        dst->limb[k] = (uint64_t)t;\n        carry = 0u;"),
    ("toy_rank_slice", "float acc = c->slots[0][(int64_t)r * h + j];", "float acc = c->slots[0][(int64_t)r * h + j] * 0.5f;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "zero_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-pthread", str(mutated), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
