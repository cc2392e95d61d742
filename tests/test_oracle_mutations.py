"""The oracle's pins must reject plausible mistakes planted in the oracle.

Each case edits one line of oracle.c (a dropped term, a wrong sign or index, a
transposed layout), builds that variant on the CPU and runs the pin suite
against it in a subprocess: the suite has to fail.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "rope_sign": ("y[i + h] = hi * c + lo * s;", "y[i + h] = hi * c - lo * s;"),
    "rope_freq": ("return pow(theta, -(2.0 * i) / d);", "return pow(theta, -(1.0 * i) / d);"),
    "rope_pairing": ("double lo = x[i], hi = x[i + h];", "double lo = x[i], hi = x[(i + 1) % d];"),
    "gqa_mapping": ("int h = j * grp + hh;\n      const uint16_t *qx = q + ((size_t)b * n_qh + h) * d;\n      for (int i = 0; i < d; ++i) xq[i] = bf16_to_double(qx[i]);\n      oracle_rope_f64(xq, d, (double)positions[b], (double)rope_theta, xq + d);\n      attend_rows(xq + d, d, (double)scale, n, kr, vr, sc,\n                  out + ((size_t)b * n_qh + h) * d);\n    }\n    free(kv);",
                    "int h = hh * n_kvh + j;\n      const uint16_t *qx = q + ((size_t)b * n_qh + h) * d;\n      for (int i = 0; i < d; ++i) xq[i] = bf16_to_double(qx[i]);\n      oracle_rope_f64(xq, d, (double)positions[b], (double)rope_theta, xq + d);\n      attend_rows(xq + d, d, (double)scale, n, kr, vr, sc,\n                  out + ((size_t)b * n_qh + h) * d);\n    }\n    free(kv);"),
    "drop_new_token": ("int n = L + 1;\n    /* dequantised", "int n = L;\n    /* dequantised"),
    "no_normalise": ("for (int i = 0; i < d; ++i) out[i] /= l;", "(void)l;"),
    "no_scale": ("sc[t] = scale * acc;", "sc[t] = acc;"),
    "pool_layout": ("return (((size_t)page * g->n_kvh + j) * g->page + off);",
                    "return (((size_t)j * g->num_pages + page) * g->page + off);"),
    "append_offset": ("int off = L % page;", "int off = (L + 1) % page;"),
    "int8_round_half_away": ("float r = rintf(t);", "float r = roundf(t);"),
    "append_unrotated": ("oracle_rope_store_f32(kx, d, positions[b], rope_theta, kr);",
                         "oracle_rope_store_f32(kx, d, 0, rope_theta, kr);"),
    "append_rotated_at_slot": ("oracle_rope_store_f32(kx, d, positions[b], rope_theta, kr);",
                               "oracle_rope_store_f32(kx, d, L, rope_theta, kr);"),
    "int8_value_from_key": ("oracle_quant_int8(vr, d, codes, &v_scales[s]);",
                            "oracle_quant_int8(kr, d, codes, &v_scales[s]);"),
    "store_fused": ("volatile float a = lc - hs, b = hc + ls;",
                    "volatile float a = fmaf(-hi, s, lo * c), b = fmaf(lo, s, hi * c);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name!r} passed every pin:\n{r.stdout[-2000:]}"
