"""The oracle's pins must catch plausible mistakes.

Each case plants one slip into a copy of the oracle source (on the CPU, in a temporary
directory), builds it, and runs the pin suite against that copy: the suite has to fail.
The real oracle is never touched.
"""
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, exact text in oracle.c, replacement)
MUTATIONS = [
    ("gemv_reversed_x", "acc += (real)row[k] * x[k];", "acc += (real)row[k] * x[K - 1 - k];"),
    ("rmsnorm_eps_outside_root", "sqrt(ss / (real)n + eps)", "(sqrt(ss / (real)n) + eps)"),
    ("rmsnorm_sum_not_mean", "sqrt(ss / (real)n + eps)", "sqrt(ss + eps)"),
    ("layernorm_unbiased_var", "sqrt(v / (real)n + eps)", "sqrt(v / (real)(n - 1) + eps)"),
    ("rope_half_sign", "? -tmp[t + half] : tmp[t - half]", "? tmp[t + half] : tmp[t - half]"),
    ("rope_pair_sign", "x[2 * j] = a * c[j] - b * s[j];", "x[2 * j] = a * c[j] + b * s[j];"),
    ("rope_freq_ladder", "pow(theta, -2.0 * (double)i / (double)d);\n        double ang = (double)pos",
     "pow(theta, -1.0 * (double)i / (double)d);\n        double ang = (double)pos"),
    ("gqa_head_modulo", "int kvh = head / group;", "int kvh = head % G;"),
    ("attn_scale_dropped", "sc[j] = p * scale;", "sc[j] = p;"),
    ("silu_sign", "g / ((real)1 + exp(-g))", "g / ((real)1 + exp(g))"),
    ("gelu_no_sqrt2", "erf(v * (real)0.70710678118654752440)", "erf(v)"),
    ("window_off_by_one", "(pos - pj < (uint32_t)window)", "(pos - pj <= (uint32_t)window)"),
    ("ring_stamp_dropped", "pr[slot] = (uint32_t)pos;", "(void)pr;"),
    ("talker_residual_dropped", "x[i] = x[i] + o[i];", "x[i] = o[i];"),
    ("layerscale_dropped", "x[i] = x[i] + (W->ls1 ? (real)W->ls1[i] * o[i] : o[i]);",
     "x[i] = x[i] + o[i];"),
    ("swiglu_operands_swapped", "silu_r(g[i]) * u[i]", "silu_r(u[i]) * g[i]"),
    ("qnorm_uses_knorm", "rms_norm_r(q + hh * d, W->q_norm", "rms_norm_r(q + hh * d, W->k_norm"),
    ("final_norm_skipped", "rms_norm_r(x, m->final_norm, h, (real)c->norm_eps, y);",
     "memcpy(y, x, sizeof(real) * (size_t)h);"),
    ("kv_append_wrong_row", "real* kd = m->kc + kv_index(m, l, s, pos);",
     "real* kd = m->kc + kv_index(m, l, s, pos > 0 ? pos - 1 : 0);"),
    ("mrope_axis_shifted", "(double)pos3[assign ? assign[i] : 0]",
     "(double)pos3[assign ? (assign[i] + 1) % 3 : 0]"),
    ("mrope_keys_turned_by_cache_position",
     "for (int gg = 0; gg < G; ++gg) rope_rotate_half_r(k + gg * d, d, cs, sn);",
     "rope_table_r(d, c->rope_theta, pos, cs, sn);\n"
     "    for (int gg = 0; gg < G; ++gg) rope_rotate_half_r(k + gg * d, d, cs, sn);"),
    ("mrope_rows_share_row0_positions", "pos3 ? pos3 + 3 * s : NULL", "pos3 ? pos3 : NULL"),
    # the flow head (Pocket TTS on wgpu, PocketFlowGpu): adaLN chunk order and wiring
    ("flow_shift_scale_swapped", "u[i] * ((real)1 + m[D + i]) + m[i];  /* modulate */",
     "u[i] * ((real)1 + m[i]) + m[D + i];  /* modulate */"),
    ("flow_modulate_one_dropped", "u[i] * ((real)1 + m[D + i]) + m[i];  /* modulate */",
     "u[i] * m[D + i] + m[i];  /* modulate */"),
    ("flow_gate_from_scale_chunk", "x[i] += m[2 * D + i] * u[i];", "x[i] += m[D + i] * u[i];"),
    ("flow_final_norm_affine", "layer_norm_r(x, one, zero, D, eps, u);",
     "layer_norm_r(x, f->ln_w[0], f->ln_b[0], D, eps, u);"),
    ("flow_final_shift_scale_swapped",
     "u[i] * ((real)1 + m[D + i]) + m[i];  /* final modulate */",
     "u[i] * ((real)1 + m[i]) + m[D + i];  /* final modulate */"),
    ("flow_bias_added_last", "real acc = (real)b[n];\n        for (int k = 0; k < K; ++k) acc += (real)row[k] * x[k];",
     "real acc = 0;\n        for (int k = 0; k < K; ++k) acc += (real)row[k] * x[k];\n        acc += (real)b[n];"),
    # the FlowLM head: the EOS logit reads the normalised row, not the residual stream
    ("eos_reads_prenorm_row", "e += (real)m->eos_w[i] * y[i];", "e += (real)m->eos_w[i] * x[i];"),
    # causal prefill: each row's key is appended before that row attends, and rows advance
    ("row_attends_before_its_key_is_appended", "pos + 1, H, G,\n                    d, att, sc);",
     "(pos > 0 ? pos : 1), H, G,\n                    d, att, sc);"),
    ("prefill_rows_share_one_position", "        m->len[stream] += 1;\n    }\n    free(buf);",
     "    }\n    m->len[stream] += n;\n    free(buf);"),
]

PIN_FILES = ["test_oracle_pins.py", "test_oracle_mrope.py"]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory() as tmp:
        mut = os.path.join(tmp, "oracle.c")
        open(mut, "w").write(src.replace(old, new))
        obuild.build(force=True, src=mut, out_dir=tmp)
        env = dict(os.environ, ORACLE_LIB_DIR=tmp)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] +
                           [os.path.join(ROOT, "tests", f) for f in PIN_FILES],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"


def test_control_unmutated_copy_passes_the_pins():
    # the same harness with no slip planted must pass, so the failures above are real catches
    with tempfile.TemporaryDirectory() as tmp:
        obuild.build(force=True, src=obuild.SRC, out_dir=tmp)
        env = dict(os.environ, ORACLE_LIB_DIR=tmp)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] +
                           [os.path.join(ROOT, "tests", f) for f in PIN_FILES],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-3000:]
