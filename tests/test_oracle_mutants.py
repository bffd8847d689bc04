"""The oracle's pins catch planted mistakes (no GPU).

Each case copies oracle/oracle.c, plants one plausible mistake in the copy
(a wrong sign, a dropped term, a transposed operand, an off-by-one, a wrong
rounding rule), builds it, and runs the pin suite against that library.  The
pin suite must fail for every mutant; a mutant that survives means some part
of the oracle is not pinned.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "bound_min_not_max": ("double t = a > bb ? a : bb;", "double t = a < bb ? a : bb;"),
    "bound_kmax_only": ("double a = qd * orc_half_to_double(kmin[(size_t)j * D + d]);",
                        "double a = qd * orc_half_to_double(kmax[(size_t)j * D + d]);"),
    "bound_group_min": ("if (s > best) best = s;", "if (s < best || h == 0) best = s;"),
    "tie_to_higher_index": ("return (a->idx > b->idx) - (a->idx < b->idx);",
                            "return (a->idx < b->idx) - (a->idx > b->idx);"),
    "topk_smallest": ("if (a->ub > b->ub) return -1;", "if (a->ub > b->ub) return 1;"),
    "recent_one_late": ("rb = (int)(start / blk);", "rb = (int)(start / blk) + 1;"),
    "sink_floor": ("int se = (sink_tokens + blk - 1) / blk;", "int se = sink_tokens / blk;"),
    "quant_half_away": ("double r = nearbyint((double)quot);", "double r = round((double)quot);"),
    "quant_scale_128": ("float s = (float)(amax / 127.0);", "float s = (float)(amax / 128.0);"),
    "quant_no_clamp_low": ("if (r < -127.0) r = -127.0;", "if (r < -128.0) r = -128.0;"),
    "quant_double_quotient": ("double r = nearbyint((double)quot);",
                              "double r = nearbyint((double)x[i] / (double)s);"),
    "append_overwrite_not_merge": ("int merge = lo < c->len;", "int merge = 0;"),
    "append_bounds_from_values": (
        "uint16_t kb = k_new[(((size_t)b * n_new + i) * c->Hkv + h) * D + d];",
        "uint16_t kb = v_new[(((size_t)b * n_new + i) * c->Hkv + h) * D + d];"),
    "f16_no_scale": ("lg[i] = scale * s;\n        if (lg[i] > M) M = lg[i];\n    }\n    double Z = 0.0;\n    for (int d = 0; d < D; ++d) out[d] = 0.0;\n    for (long i = 0; i < n; ++i) {\n        double w = exp(lg[i] - M);\n        Z += w;\n        const uint16_t",
                     "lg[i] = s;\n        if (lg[i] > M) M = lg[i];\n    }\n    double Z = 0.0;\n    for (int d = 0; d < D; ++d) out[d] = 0.0;\n    for (long i = 0; i < n; ++i) {\n        double w = exp(lg[i] - M);\n        Z += w;\n        const uint16_t"),
    "f16_keys_as_values": ("const uint16_t *v = V + (size_t)tok[i] * D;",
                           "const uint16_t *v = K + (size_t)tok[i] * D;"),
    "int8_no_kscale": ("lg[i] = (double)dot * (double)q_scale * (double)ks[tok[i]] * scale;",
                       "lg[i] = (double)dot * (double)q_scale * scale;"),
    "int8_no_vscale": ("double sv = (double)vs[tok[i]];", "double sv = 1.0;"),
    "int8_vscale_from_k": ("double sv = (double)vs[tok[i]];", "double sv = (double)ks[tok[i]];"),
    "gqa_modulo_mapping": ("const float *qh = q + ((size_t)b * H + (size_t)g * G + hh) * D;",
                           "const float *qh = q + ((size_t)b * H + (size_t)g + hh) * D;"),
    "gqa_modulo_mapping_select": (
        "int b = p / c->Hkv, g = p % c->Hkv;\n        const float *qg = q + ((size_t)b * H + (size_t)g * G) * D;",
        "int b = p / c->Hkv, g = p % c->Hkv;\n        const float *qg = q + ((size_t)b * H + (size_t)g) * D;"),
    "partial_block_overrun": ("t < (long)(sel[i] + 1) * blk && t < L; ++t)",
                              "t < (long)(sel[i] + 1) * blk; ++t)"),
    "half_subnormal_exp": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    # sparse-V (eps mode)
    "sv_one_scope_for_all": ("while (j < n && tok[j] / ORC_SV_CHUNK == tok[i] / ORC_SV_CHUNK) ++j;",
                             "while (j < n) ++j;"),
    "sv_le_not_lt": ("keep[u] = !(exp(lg[u] - m) < thr);", "keep[u] = !(exp(lg[u] - m) <= thr);"),
    "sv_sum_not_mean": ("double thr = eps * sum / (double)(j - i);", "double thr = eps * sum;"),
    "sv_dropped_out_of_denominator": (
        "            Zd += w;\n            continue;\n        }\n        const uint16_t *vr",
        "            Zd += w;\n            Z -= w;\n            continue;\n        }\n        const uint16_t *vr"),
    # q8_0
    "half_round_down": ("double n = nearbyint(ldexp(a, 10 - e));", "double n = floor(ldexp(a, 10 - e));"),
    "q8_codes_from_unrounded_scale": ("double dg = orc_half_to_double(d[g]);", "double dg = (double)s32;"),
    "q8_amax_of_first_group": ("double a = fabs((double)xg[i]);", "double a = fabs((double)x[i]);"),
    "q8_logit_group0_scale": ("acc += orc_half_to_double(kd[(size_t)tok[i] * ng + g]) * (double)dot;",
                              "acc += orc_half_to_double(kd[(size_t)tok[i] * ng]) * (double)dot;"),
    "q8_value_scale_wrong_group": (
        "out[d] += w * orc_half_to_double(vd[(size_t)tok[i] * ng + d / ORC_QGROUP]) *",
        "out[d] += w * orc_half_to_double(vd[(size_t)tok[i] * ng + (d / ORC_QGROUP + 1) % ng]) *"),
    # q4_0
    "q4_scale_positive": ("float s32 = (float)(m / -8.0);", "float s32 = (float)(m / 8.0);"),
    "q4_max_by_value": ("            if (mag > amax) {\n                amax = mag;\n                m = (double)xg[i];",
                        "            if (mag > amax) {\n                amax = mag;\n                m = fabs((double)xg[i]);"),
    "q4_nibbles_swapped": ("packed[g * (ORC_QGROUP / 2) + i] = (uint8_t)(c4[2 * i] | (c4[2 * i + 1] << 4));",
                           "packed[g * (ORC_QGROUP / 2) + i] = (uint8_t)(c4[2 * i + 1] | (c4[2 * i] << 4));"),
    "q4_no_offset_in_dot": ("dot += (int64_t)qc[c] * (int64_t)(q4_code(k, c) - 8);",
                            "dot += (int64_t)qc[c] * (int64_t)q4_code(k, c);"),
    "q4_round_half_up": ("double r4 = nearbyint((double)qt) + 8.0;", "double r4 = floor((double)qt + 0.5) + 8.0;"),
    # moment tail (R10)
    "tail_without_count": ("x[n] = scale * s + log((double)mj);", "x[n] = scale * s;"),
    "tail_full_block_count": ("x[n] = scale * s + log((double)mj);",
                              "x[n] = scale * s + log((double)blk);"),
    "tail_without_scale": ("x[n] = scale * s + log((double)mj);", "x[n] = s + log((double)mj);"),
    "tail_ignores_listing": ("if (sel[i] >= 0 && sel[i] < nb) listed[sel[i]] = 1;",
                             "if (sel[i] >= 0 && sel[i] < nb) listed[sel[i]] = 0;"),
    "tail_value_is_key_mean": (
        "tail_val[(size_t)j * D + d] = orc_half_to_double(mV[(size_t)j * D + d]);",
        "tail_val[(size_t)j * D + d] = orc_half_to_double(mK[(size_t)j * D + d]);"),
    "moment_divides_by_blk": ("mean[(size_t)j * D + d] = orc_double_to_half(sum / (double)m);",
                              "mean[(size_t)j * D + d] = orc_double_to_half(sum / (double)blk);"),
    "moment_skips_first_row": ("for (int t = lo; t < lo + m; ++t) sum += X[(size_t)t * D + d];",
                               "for (int t = lo + 1; t < lo + m; ++t) sum += X[(size_t)t * D + d];"),
    # f32 append input (R11)
    "f32_bounds_to_nearest": ("uint16_t dn = orc_double_to_half_dir(xmin, -1);",
                              "uint16_t dn = orc_double_to_half(xmin);"),
    "f32_bounds_overwrite": ("int held = first < c->len;", "int held = 0;"),
    "half_dir_wrong_step": ("if (neg == toward_pos) return (uint16_t)(h - 1);",
                            "if (neg == toward_pos) return (uint16_t)(h + 1);"),
    "f32_values_as_keys": ("orc_quantize_row(vx, D, (int8_t *)c->V + r * D, &c->vs[r]);",
                           "orc_quantize_row(kx, D, (int8_t *)c->V + r * D, &c->vs[r]);"),
}


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: snippet not found exactly once"
    mdir = os.path.join(tmp, name)
    os.makedirs(mdir)
    cfile = os.path.join(mdir, "oracle.c")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(mdir, "liboracle.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", lib, cfile, "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_sparse_v.py"),
                        os.path.join(ROOT, "tests", "test_oracle_q8_0.py"),
                        os.path.join(ROOT, "tests", "test_oracle_q4_0.py"),
                        os.path.join(ROOT, "tests", "test_oracle_tail.py"),
                        os.path.join(ROOT, "tests", "test_oracle_append_f32.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_is_caught():
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            res = list(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp), MUTANTS.items()))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    survivors = [n for n, rc in res if rc == 0]
    assert not survivors, f"pins missed planted mistakes: {survivors}"
    # a crash is not a catch: the suite must have run and failed
    assert all(rc == 1 for _, rc in res), res
