"""Plant plausible slips in copies of the oracle and check that the pins catch each one.

Each mutant is oracle.c with one textual edit (a dropped term, a flipped sign,
a wrong index or a swapped operand), compiled into a temporary library.  The
real oracle passes every pin (test_oracle_pins.py); every mutant must fail at
least one.
"""

import shutil
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "rms_drops_eps": ("double inv = 1.0 / sqrt(ms + eps);", "double inv = 1.0 / sqrt(ms);"),
    "rms_wrong_mean": ("double ms = ss / (double)D;", "double ms = ss / (double)(D - 1);"),
    "rms_drops_weight": ("yr[d] = xr[d] * inv * w[d];", "yr[d] = xr[d] * inv;"),
    "rope_sign": ("yr[2 * i] = a * c - b * sn;", "yr[2 * i] = a * c + b * sn;"),
    "rope_pair_index": ("double c = cos_tab[s * P + i], sn = sin_tab[s * P + i];",
                        "double c = cos_tab[s * P + (P - 1 - i)], sn = sin_tab[s * P + (P - 1 - i)];"),
    "rope_half_split": ("double a = xr[2 * i], b = xr[2 * i + 1];", "double a = xr[i], b = xr[i + P];"),
    "attn_drops_scale": ("sc[j] = scale * dot;", "sc[j] = dot;"),
    "attn_k_is_v": ("const double *kr = k + ((b * Skv + kv_begin + j) * H + h) * D;\n                double dot",
                    "const double *kr = v + ((b * Skv + kv_begin + j) * H + h) * D;\n                double dot"),
    "attn_lse_drops_max": ("lse[(b * H + h) * nrows + r] = m + log(l);", "lse[(b * H + h) * nrows + r] = log(l);"),
    "attn_no_normalise": ("for (int64_t d = 0; d < D; ++d) orow[d] /= l;", ""),
    "attn_ignores_begin": ("const double *vr = v + ((b * Skv + kv_begin + j) * H + h) * D;",
                           "const double *vr = v + ((b * Skv + j) * H + h) * D;"),
    "causal_strict": ("if (causal) nv = qi - kv_begin + 1 < n ? qi - kv_begin + 1 : n;",
                      "if (causal) nv = qi - kv_begin < n ? qi - kv_begin : n;"),
    "causal_ignores_begin": ("if (causal) nv = qi - kv_begin + 1 < n ? qi - kv_begin + 1 : n;",
                             "if (causal) nv = qi + 1 < n ? qi + 1 : n;"),
    "ln_unbiased_var": ("const double inv = 1.0 / sqrt(ss / (double)C + eps);",
                        "const double inv = 1.0 / sqrt(ss / (double)(C - 1) + eps);"),
    "ln_scale_not_plus_one": ("yr[c] = (xr[c] - mu) * inv * (1.0 + sc) + sh;", "yr[c] = (xr[c] - mu) * inv * sc + sh;"),
    "e4m3_bias8": ("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3_ties_odd": ("(err == best_err && (c & 1) == 0 && (best & 1) == 1)", "(err == best_err && (c & 1) == 1)"),
    "quant_scale_127": ("float sc = amax > 0.0f ? amax / 448.0f : 1.0f;", "float sc = amax > 0.0f ? amax / 127.0f : 1.0f;"),
    "gemm_drops_b_scale": ("out[m * N + n] = acc * (double)a_scale[m] * (double)b_scale[n];",
                           "out[m * N + n] = acc * (double)a_scale[m];"),
    "merge_weight_vs_max": ("double wgt = exp(lse_parts[c * part_l + li] - L);",
                            "double wgt = exp(lse_parts[c * part_l + li] - mx);"),
    "merge_lse_drops_max": ("double L = mx + log(sum);", "double L = log(sum);"),
    "merge_uniform": ("double wgt = exp(lse_parts[c * part_l + li] - L);", "double wgt = 1.0 / (double)C;"),
}


@pytest.fixture(scope="module")
def src():
    return oracle.SOURCE.read_text()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src, tmp_path):
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(path), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
