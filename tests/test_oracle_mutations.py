"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in a copy of the oracle: a wrong bias, tie
rule or sign in a number format, a wrong index, stride, head mapping or
scale in the cache write, the MLA assembly, decode attention or the MLA
chain, a dropped term, an off-by-one in the causal position.  It then runs
every pin in tests/test_oracle_*.py against that copy
(tests/oracle_pin_battery.py, in a child process) and requires at least two
pins to fail, so that no mistake rests on a single pin.  The unmodified
copy must pass every pin.  The mistakes keep every access in bounds, so a
failing pin, not a crash, is what catches them.
"""
import json
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (id, file in oracle/, text that occurs exactly once, replacement)
MUTATIONS = [
    # number formats
    ("e4m3_bias", "oracle.c", "F_E4M3 = {4, 3, 7, 0,", "F_E4M3 = {4, 3, 8, 0,"),
    ("ties_to_odd", "oracle.c", "else code = (lo & 1u) ? lo + 1u : lo;",
     "else code = (lo & 1u) ? lo : lo + 1u;"),
    ("e4m3_overflow_to_nan", "oracle.c", "code = top; /* saturate */",
     "code = f->nan_code; /* saturate */"),
    ("subnormal_exponent", "oracle.c", "return ldexp((double)mant, 1 - f->bias - f->m);",
     "return ldexp((double)mant, 0 - f->bias - f->m);"),
    ("negative_zero_sign", "oracle.c", "uint32_t sign = signbit(y) ? sign_bit : 0u;",
     "uint32_t sign = (y < 0) ? sign_bit : 0u;"),
    ("nan_to_inf", "oracle.c", "if (isnan(y)) return f->nan_code;",
     "if (isnan(y)) return f->inf_code;"),
    ("overflow_tie_to_finite", "oracle.c", "if (a < mid) code = top;",
     "if (a <= mid) code = top;"),
    # cache write
    ("swa_table_ignored", "oracle.c", "    s = swa[s];\n", "    s = s;\n"),
    ("scale_skipped_for_same_format", "oracle.c",
     "const int raw = (src_dtype == cache_dtype) && k_scale == NULL;",
     "const int raw = (src_dtype == cache_dtype);"),
    ("head_dim_transposed", "oracle.c",
     "int64_t dst = block_idx * block_stride + block_offset * row + (int64_t)h * head_size + i;",
     "int64_t dst = block_idx * block_stride + block_offset * row + (int64_t)i * num_heads + h;"),
    ("scale_multiplied", "oracle.c", "if (k_scale) kx = kx / *k_scale;",
     "if (k_scale) kx = kx * *k_scale;"),
    ("v_divided_by_k_scale", "oracle.c", "if (v_scale) vx = vx / *v_scale;",
     "if (v_scale) vx = vx / *k_scale;"),
    # MLA K assembly
    ("rope_over_nope", "oracle.c",
     "int64_t to = n * k_stride0 + (int64_t)h * k_stride1 + nope_dim + i;",
     "int64_t to = n * k_stride0 + (int64_t)h * k_stride1 + i;"),
    ("nope_of_head0", "oracle.c",
     "int64_t from = n * nope_stride0 + (int64_t)h * nope_stride1 + i;",
     "int64_t from = n * nope_stride0 + i;"),
    # decode attention
    ("q_row_of_kv_head", "oracle.c",
     "qd[i] = load_elem(q_dtype, q, ((int64_t)b * num_q_heads + h) * d + i);",
     "qd[i] = load_elem(q_dtype, q, ((int64_t)b * num_q_heads + g) * d + i);"),
    ("scale_dropped", "oracle.c", "    s[j] = scale * dot;", "    s[j] = dot;"),
    ("weights_unnormalised", "oracle.c", "    double p = exp(s[j] - smax) / l;\n    ps += p;",
     "    double p = exp(s[j] - smax);\n    ps += p;"),
    ("gqa_interleaved", "oracle.c", "const int32_t g = h / group;",
     "const int32_t g = h % num_kv_heads;"),
    ("rows_reversed_in_block", "oracle.c",
     "int64_t phys_row = blk * block_size + j % block_size;",
     "int64_t phys_row = blk * block_size + (block_size - 1 - j % block_size);"),
    ("v_dequantised_by_k_scale", "oracle.c",
     "V[n * d + i] = load_elem(cache_dtype, v_cache, base + i) * (double)v_scale;",
     "V[n * d + i] = load_elem(cache_dtype, v_cache, base + i) * (double)k_scale;"),
    ("lse_without_max", "oracle.c", "  if (lse) *lse = smax + log(l);\n  if (psum)",
     "  if (lse) *lse = log(l);\n  if (psum)"),
    # MLA chain
    ("absorb_head_stride_dropped", "oracle.c",
     "load_elem(w_dtype, w_uk, (int64_t)c * wcols + (int64_t)h * d_h + i)",
     "load_elem(w_dtype, w_uk, (int64_t)c * wcols + (int64_t)h + i)"),
    ("rope_score_term_dropped", "oracle.c",
     "for (int32_t i = 0; i < dk; ++i) dot += qd[i] * R[j * dk + i];",
     "for (int32_t i = 0; i < d_c; ++i) dot += qd[i] * R[j * dk + i];"),
    ("project_all_heads_head0", "oracle.c",
     "load_elem(w_dtype, w_uv, (int64_t)c * wcols + (int64_t)h * d_v + i)",
     "load_elem(w_dtype, w_uv, (int64_t)c * wcols + i)"),
    ("mla_lse_without_max", "oracle.c", "  if (lse) *lse = smax + log(l);\n  free(qd); free(R);",
     "  if (lse) *lse = log(l);\n  free(qd); free(R);"),
    # MLA in the pages' explicit form
    ("explicit_wuv_of_head0", "oracle.c",
     "load_elem(w_dtype, w_uv, (int64_t)k * num_heads * d_v + (int64_t)h * d_v + i);",
     "load_elem(w_dtype, w_uv, (int64_t)k * num_heads * d_v + i);"),
    ("explicit_rope_dropped", "oracle.c",
     "for (int32_t r = 0; r < d_r; ++r) K[n * dk + d_h + r] = c[d_c + r];",
     "for (int32_t r = 0; r < d_r; ++r) K[n * dk + d_h + r] = 0.0;"),
    ("explicit_wuk_head_stride_dropped", "oracle.c",
     "load_elem(w_dtype, w_uk, (int64_t)k * num_heads * d_h + (int64_t)h * d_h + i);",
     "load_elem(w_dtype, w_uk, (int64_t)k * num_heads * d_h + (int64_t)h + i);"),
    # causal prefill position
    ("prefill_position_off_by_one", "__init__.py", "p = int(context_lens[b]) - n + j\n",
     "p = int(context_lens[b]) - n + j - 1\n"),
]


def _run_battery(tmp, mutation):
    d = os.path.join(tmp, mutation[0] if mutation else "control")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    if mutation:
        _, fname, find, repl = mutation
        path = os.path.join(d, "oracle", fname)
        with open(path) as f:
            src = f.read()
        assert src.count(find) == 1, f"{mutation[0]}: the text to mutate must occur once"
        with open(path, "w") as f:
            f.write(src.replace(find, repl))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "oracle_pin_battery.py"), d],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    cases = [None] + MUTATIONS
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        outs = list(ex.map(lambda m: _run_battery(tmp, m), cases))
    return {("control" if m is None else m[0]): o for m, o in zip(cases, outs)}


def test_unmodified_oracle_passes_every_pin(results):
    r = results["control"]
    assert r["ran"] >= 80 and r["failed"] == [], r["failed"]


@pytest.mark.parametrize("mid", [m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(results, mid):
    r = results[mid]
    # every planted mistake fails at least two independent pins
    assert len(r["failed"]) >= 2, (mid, r["failed"])
