"""The oracle's pins must catch plausible mistakes (CPU only).

Each case plants one mistake (a dropped term, a wrong sign or index, a
transposed or swapped operand) in a temporary copy of ``oracle.c``, builds
it, points the ``oracle`` module at that build and runs every pin of
``test_oracle_ops`` and ``test_oracle_model``: at least one must fail.  The
committed oracle source is never modified.
"""
import inspect
import subprocess

import pytest

import oracle
import synth
from tests import test_oracle_model as tm
from tests import test_oracle_ops as to

MUTANTS = {
    "rmsnorm_drops_eps": ("ss / (double)n + eps", "ss / (double)n"),
    "rmsnorm_sum_not_mean": ("ss / (double)n + eps", "ss + eps"),
    "rmsnorm_drops_gain": ("y[i] = x[i] * r * orc_bf16_to_double(gain[i]);", "y[i] = x[i] * r;"),
    "gemv_transposed": ("acc += orc_bf16_to_double(w[i]) * hd[i];",
                        "acc += orc_bf16_to_double(((const uint16_t *)W)[((size_t)i * rows + o) % ((size_t)rows * K)]) * hd[i];"),
    "gemv_int8_wrong_row_scale": ("y[o] = (double)scales[o] * acc;", "y[o] = (double)scales[0] * acc;"),
    "rope_wrong_sign": ("u[i] = a * c - b * s;", "u[i] = a * c + b * s;"),
    "rope_wrong_frequency": ("-2.0 * (double)i / (double)d", "-1.0 * (double)i / (double)d"),
    "rope_adjacent_pairs": ("double a = u[i], b = u[i + half];\n        u[i] = a * c - b * s;\n        u[i + half] = b * c + a * s;",
                            "double a = u[2 * i], b = u[2 * i + 1];\n        u[2 * i] = a * c - b * s;\n        u[2 * i + 1] = b * c + a * s;"),
    "attention_drops_scale": ("s[m] = acc * scale;", "s[m] = acc;"),
    "attention_k_for_v": ("acc += s[m] * orc_bf16_to_double(Vc[(size_t)m * d + i]);",
                          "acc += s[m] * orc_bf16_to_double(Kc[(size_t)m * d + i]);"),
    "attention_excludes_new_token": ("orc_attention(p + 1, d,", "orc_attention(p, d,"),
    "gqa_wrong_head_map": ("int g = j / G;", "int g = j % nkv;"),
    "cache_stores_v_as_k": ("kcache[(row + p) * d + i] = orc_double_to_bf16(k[(size_t)g * d + i]);",
                            "kcache[(row + p) * d + i] = orc_double_to_bf16(v[(size_t)g * d + i]);"),
    "k_not_rotated": ("for (int g = 0; g < nkv; ++g) orc_rope(d, p, c->rope_theta, k + (size_t)g * d);", ""),
    "attn_residual_dropped": ("mat_vec(c, 0, H, nq * d, w->wo, w->so, ob, y);\n    for (int i = 0; i < H; ++i) x[i] += y[i];",
                              "mat_vec(c, 0, H, nq * d, w->wo, w->so, ob, y);\n    for (int i = 0; i < H; ++i) x[i] = y[i];"),
    "gemv_int4_high_nibble_first": ("const int u = (w[i / 2] >> (4 * (i & 1))) & 15;",
                                    "const int u = (w[i / 2] >> (4 * (1 - (i & 1)))) & 15;"),
    "gemv_int4_one_scale_per_row": ("tot += (double)scales[(size_t)o * ng + g] * acc;",
                                    "tot += (double)scales[(size_t)o * ng] * acc;"),
    "gemv_int4_no_zero_point": ("acc += (double)(u - 8) * hd[i];", "acc += (double)u * hd[i];"),
    "swiglu_gate_up_swapped": ("orc_silu(gt[i]) * up[i]", "orc_silu(up[i]) * gt[i]"),
    "silu_wrong_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "norm_gains_swapped": ("orc_rmsnorm(H, x, w->attn_norm, c->rms_eps, y);", "orc_rmsnorm(H, x, w->mlp_norm, c->rms_eps, y);"),
    "bf16_truncates": ("double v = ldexp(nearbyint(ldexp(m, 8)), e - 8);", "double v = ldexp(trunc(ldexp(m, 8)), e - 8);"),
    "argmax_highest_index_on_tie": ("if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;"),
    "final_norm_skipped": ("orc_rmsnorm(H, x, wt->final_norm, c->rms_eps, y);",
                           "for (int i = 0; i < H; ++i) y[i] = x[i] * orc_bf16_to_double(wt->final_norm[i]);"),
}


def _pins():
    out = []
    for mod in (to, tm):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if name.startswith("test_") and fn.__module__ == mod.__name__:
                out.append(fn)
    return out


def _tiny():
    wl = synth.workload("tiny")
    return wl, tm.with_random_gains(synth.make_model(wl, seed=1))


def _failing_pins(tiny):
    failed = []
    for fn in _pins():
        args = [tiny] if "tiny" in inspect.signature(fn).parameters else []
        try:
            fn(*args)
        except (AssertionError, ValueError):
            failed.append(fn.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found exactly once: %s" % name
    (tmp_path / "oracle_mut.c").write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", str(tmp_path / "oracle_mut.c"),
                           "-o", str(so), "-lm"])
    oracle.use_library(oracle.load(str(so)))
    try:
        failed = _failing_pins(_tiny())
    finally:
        oracle.use_library(None)
    assert failed, "no pin caught the planted mistake %r" % name


def test_unmutated_oracle_passes_every_pin():
    assert _failing_pins(_tiny()) == []
