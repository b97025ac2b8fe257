"""The layer pins catch plausible mistakes (CPU): each case plants one mistake in a private copy
of the oracle (its C file or its Python compositions), loads that copy as a separate module and
checks that the named pins fail on it while an unmodified copy passes them all. Nothing here
touches the repository's oracle."""
import importlib.util
import os
import shutil

import pytest

import oracle as orc

from _layer_pins import PINS

ORACLE_DIR = os.path.dirname(os.path.abspath(orc.__file__))

# (file, original text, planted mistake, pins that must fail)
MUTATIONS = {
    "rope_exponent_halved": ("orc.c", "pow(theta, -2.0 * (double)i / (double)hd)",
                             "pow(theta, -1.0 * (double)i / (double)hd)", ["rope_frequency"]),
    "attention_scale_1_over_hd": ("orc.c", "double scale = 1.0 / sqrt((double)hd);", "double scale = 1.0 / (double)hd;",
                                  ["attention_scale"]),
    "attention_scale_dropped": ("orc.c", "double scale = 1.0 / sqrt((double)hd);", "double scale = 1.0;",
                                ["attention_scale"]),
    "rmsnorm_weight_dropped": ("orc.c", "out[r * k + i] = xr[i] * rstd * (w ? (double)w[i] : 1.0);",
                               "out[r * k + i] = xr[i] * rstd;",
                               ["layer_attention_half", "layer_ffn_half", "head_out_norm"]),
    "o_residual_dropped": ("__init__.py", 'x = x + qgemm(TYPE_Q4_K, lw["wo"], q2, d2)',
                           'x = qgemm(TYPE_Q4_K, lw["wo"], q2, d2)', ["layer_residuals", "layer_attention_half"]),
    "down_residual_dropped": ("__init__.py", 'x = x + qgemm(TYPE_Q6_K, lw["wdown"], q4, d4)',
                              'x = qgemm(TYPE_Q6_K, lw["wdown"], q4, d4)', ["layer_residuals", "layer_ffn_half"]),
    "o_fed_by_residual": ("__init__.py", 'ex["attn_out"] = o\n    q2, d2, _ = quantize_act(o)',
                          'ex["attn_out"] = o\n    q2, d2, _ = quantize_act(x)',
                          ["layer_attention_half"]),
    "attn_norm_dropped": ("__init__.py", 'q1, d1, _ = quantize_act(x, lw["attn_norm"], eps)',
                          "q1, d1, _ = quantize_act(x, None, eps)", ["layer_attention_half"]),
    "ffn_norm_swapped": ("__init__.py", 'ex["x_mid"] = x\n    q3, d3, _ = quantize_act(x, lw["ffn_norm"], eps)',
                         'ex["x_mid"] = x\n    q3, d3, _ = quantize_act(x, lw["attn_norm"], eps)', ["layer_ffn_half"]),
    "swiglu_operands_swapped": ("__init__.py", "h = swiglu(g, u)", "h = swiglu(u, g)", ["layer_ffn_half"]),
    "head_out_norm_dropped": ("__init__.py", "q, d, _ = quantize_act(hidden_rows, out_norm, eps)",
                              "q, d, _ = quantize_act(hidden_rows, None, eps)", ["head_out_norm"]),
}


def _oracle_copy(tmp_path, name, mutation=None):
    d = tmp_path / name
    d.mkdir()
    orc.build()  # the repository's library is current, so a Python-only copy can reuse it
    shutil.copy2(os.path.join(ORACLE_DIR, "orc.c"), d / "orc.c")
    shutil.copy2(os.path.join(ORACLE_DIR, "__init__.py"), d / "__init__.py")
    if mutation is not None:
        fname, old, new, _ = mutation
        path = d / fname
        src = path.read_text()
        assert src.count(old) == 1, f"{name}: the text to mutate must occur exactly once in {fname}"
        path.write_text(src.replace(old, new))
    if mutation is None or mutation[0] != "orc.c":
        shutil.copy2(os.path.join(ORACLE_DIR, "liborc.so"), d / "liborc.so")
    spec = importlib.util.spec_from_file_location(f"oracle_copy_{name}", d / "__init__.py",
                                                  submodule_search_locations=[str(d)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_unmodified_copy_passes_every_pin(tmp_path):
    mod = _oracle_copy(tmp_path, "plain")
    for pin in PINS.values():
        pin(mod)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    mod = _oracle_copy(tmp_path, name, MUTATIONS[name])
    for pin in MUTATIONS[name][3]:
        with pytest.raises(AssertionError):
            PINS[pin](mod)
