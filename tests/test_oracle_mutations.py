"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case compiles a copy of oracle/attn_oracle.c with one plausible mistake
(a dropped term, a wrong sign, a wrong index, a swapped operand), swaps it in
for the real oracle, and runs the pin tests of test_oracle.py against it: at
least one pin must fail.  The real oracle is restored afterwards.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTATIONS = {
    "head_mapping_modulo": ("int kh = h / pr->group;",
                            "int kh = h % (pr->num_q_heads / pr->group);"),
    "scale_dropped": ("s[j] = pr->scale * acc;", "s[j] = acc;"),
    "softmax_sign_flipped": ("double w = exp(s[j] - M);", "double w = exp(M - s[j]);"),
    "causal_off_by_one": ("int64_t lim = L - n + i + 1;", "int64_t lim = L - n + i;"),
    "sink_left_out_of_normaliser": ("double Z = exp(t - M);", "double Z = 0.0;"),
    "page_index_swapped": ("page = kv->page_table[(int64_t)b * kv->max_pages + t / kv->page_size];",
                           "page = kv->page_table[(int64_t)b * kv->max_pages + t % kv->page_size];"),
    "lse_without_log": ("a->lse[item] = M + log(Z);", "a->lse[item] = M + Z;"),
    "v_read_from_k": ("const uint16_t *vp = kv_row(pr->v, b, j, kh);\n        Z += 0;",
                      None),
    "partial_max_unscaled": ("double w = exp(s[j] - m);", "double w = exp(s[j]);"),
    "sparse_batch_offset_dropped": ("int64_t r = kv->indices[(int64_t)b * kv->indices_stride + t];",
                                    "int64_t r = kv->indices[t];"),
    "sparse_slot_page_swapped": ("slot = r % kv->page_size;\n    } else if",
                                 "slot = r / kv->page_size;\n    } else if"),
    "last_key_dropped": ("for (int64_t j = 0; j < nvis; ++j) {\n        double w",
                         "for (int64_t j = 0; j + 1 < nvis; ++j) {\n        double w"),
    # the error-bound statistics (oracle_spread)
    "spread_weights_unnormalised": ("double w = exp(s[j] - M) / Z;", "double w = exp(s[j] - M);"),
    "spread_sqrt_dropped": ("sd[c] = sqrt(sd[c]);", "sd[c] = sd[c];"),
    "spread_centre_dropped": ("double d = bf16_to_double(vp[c]) - am[c];",
                              "double d = bf16_to_double(vp[c]);"),
    "spread_abs_dropped": ("am[c] += w * fabs(bf16_to_double(vp[c]));",
                           "am[c] += w * bf16_to_double(vp[c]);"),
}
# v_read_from_k: replace only in the full-attention item
MUTATIONS["v_read_from_k"] = ("        Z += w;\n        const uint16_t *vp = kv_row(pr->v, b, j, kh);",
                              "        Z += w;\n        const uint16_t *vp = kv_row(pr->k, b, j, kh);")

RUNNER = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import test_oracle_mutations as m
oracle.use_library({lib!r})
failed = m.run_pins()
print("FAILED:" + ",".join(failed))
sys.exit(0 if failed else 3)
"""


def run_pins():
    from tests import test_oracle as pins
    failed = []
    for name in [n for n in dir(pins) if n.startswith("test_")]:
        fn = getattr(pins, name)
        params = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        cases = [{}]
        if params:
            argnames, values = params[0].args
            argnames = [a.strip() for a in argnames.split(",")]
            cases = [dict(zip(argnames, vals)) for vals in values]
        for kw in cases:
            try:
                fn(**kw)
            except AssertionError:
                failed.append(name)
                break
    return failed


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path):
    """The mutant runs in a child process: a mistake that makes the oracle
    read out of bounds and crash counts as caught too."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTATIONS[mutation]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor not found: {mutation}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c", RUNNER.format(root=root, lib=lib)],
                          capture_output=True, text=True, timeout=600, cwd=root)
    assert proc.returncode != 3, f"no pin caught the planted mistake {mutation}"
    if proc.returncode == 0:
        assert "FAILED:" in proc.stdout and proc.stdout.strip() != "FAILED:"
