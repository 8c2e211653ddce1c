"""Planted mistakes in the oracle must each fail at least one pin (no GPU).

Each mutant is a copy of ``oracle/msa_oracle.c`` with one plausible mistake (a
flipped sign, a dropped term, a wrong index, a wrong rounding), compiled on the
CPU into a temporary directory and loaded, in a child process, in place of the
real build while the pins run.  A mutant that writes out of bounds may crash its
child; that counts as caught.  The real oracle source is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "rope_sign": ("y[iu] = u * c - v * s;", "y[iu] = u * c + v * s;"),
    "rope_pairing": ("int32_t iv = (style == ORACLE_ROPE_GPTJ) ? 2 * k + 1 : k + half;",
                     "int32_t iv = (style == ORACLE_ROPE_GPTJ) ? 2 * k + 1 : rd - 1 - k;"),
    "rope_frequency": ("2.0 * (double)k / (double)rd", "(double)k / (double)rd"),
    "rms_mean_dropped": ("ss / (float)D + eps", "ss + eps"),
    "rms_weight_reversed": ("(w ? w[i] : 1.0f)", "(w ? w[D - 1 - i] : 1.0f)"),
    "e4m3_ties_away": ("float n = rintf(ldexpf(a, 3 - E));", "float n = roundf(ldexpf(a, 3 - E));"),
    "e4m3_overflow_to_nan": ("if (a >= 448.0f)\n        return sign | 0x7E;",
                             "if (a > 448.0f)\n        return 0x7F;"),
    "e4m3_subnormal_scale": ("float n = rintf(ldexpf(a, 9));", "float n = rintf(ldexpf(a, 8));"),
    "bf16_ties_up": ("dropped > 0x8000u ||", "dropped >= 0x8000u ||"),
    "place_page_bound": ("if (pg < 0 || pg >= num_pages)", "if (pg < 0 || pg > num_pages)"),
    "place_offset": ("*off = ls % P;", "*off = (ls + 1) % P;"),
    "place_table_bound": ("if (block >= page_table_len)", "if (block > page_table_len)"),
    "scale_multiplied": ("1.0f / cache_scale(sh, scales, 1, h)", "cache_scale(sh, scales, 1, h)"),
    "v_gets_normalised": ("store_cache_row(v_cache, page, h, off, x, D,",
                          "oracle_rmsnorm(x, w[1], D, sh->rms_eps, x);\n"
                          "                store_cache_row(v_cache, page, h, off, x, D,"),
    "idx_section_offset": ("const int64_t off_iq = off_v + (int64_t)Hkv * D;",
                           "const int64_t off_iq = off_k + (int64_t)Hkv * D;"),
    "k_weight_swapped": ("oracle_rmsnorm(x, w[1], D, sh->rms_eps, y);",
                         "oracle_rmsnorm(x, w[0], D, sh->rms_eps, y);"),
    "stride_head_token_swapped": ("head * c->stride_head + off * c->stride_token",
                                  "head * c->stride_token + off * c->stride_head"),
    "indexer_block_size": ("const int64_t b = j / block_tokens;", "const int64_t b = j / (block_tokens + 1);"),
    "indexer_visibility": ("for (int64_t j = 0; j < L; ++j) {", "for (int64_t j = 0; j <= L; ++j) {"),
    "indexer_ties_high": ("if (best < 0 || bs[b] > bs[best])", "if (best < 0 || bs[b] >= bs[best])"),
    "indexer_scale_dropped": ("oracle_e4m3_decode(idx_k_cache->data[e + d]) * k_scale", "oracle_e4m3_decode(idx_k_cache->data[e + d])"),
    "indexer_table_offset": ("const int64_t ti = table_offset[t] + j / P;", "const int64_t ti = j / P;"),
    "projection_weight_transposed": ("projection_operand(hw, dtype, j * weight_stride + k)",
                                     "projection_operand(hw, dtype, k * weight_stride + j)"),
    "projection_dropped_term": ("for (int64_t k = 0; k < hidden_size; ++k)",
                                "for (int64_t k = 1; k < hidden_size; ++k)"),
    "projection_fp32_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "projection_hidden_stride": ("projection_operand(hx, dtype, t * hidden_stride + k)",
                                 "projection_operand(hx, dtype, t * hidden_size + k)"),
    "projection_weight_scale_by_token": ("(double)weight_scales[j]", "(double)weight_scales[t % width]"),
    "projection_scale_dropped": ("(float)(acc * sx * sw)", "(float)(acc * sx)"),
    "projection_e4m3_as_bf16": ("if (dtype == ORACLE_DTYPE_E4M3)\n        return (double)oracle_e4m3_decode",
                                "if (dtype != ORACLE_DTYPE_E4M3)\n        return (double)oracle_e4m3_decode"),
    "indexer_sum_heads": ("                if (s > bs[b])\n                    bs[b] = s;", "                bs[b] = (bs[b] == -INFINITY ? 0.0f : bs[b]) + s;"),
}


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "msa_oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(src), "-lm"], check=True)
    runner = (
        "import sys, oracle, oracle_pins\n"
        "oracle._lib = oracle.load(sys.argv[1])\n"
        "failed = []\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin()\n"
        "    except Exception:\n"
        "        failed.append(pin.__name__)\n"
        "print(' '.join(failed))\n"
        "sys.exit(0 if failed else 3)\n")
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([here, os.path.dirname(here), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", runner, str(so)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 3, f"no pin caught mutant {name}"
