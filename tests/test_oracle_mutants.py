"""Plant plausible mistakes in copies of the oracle's C source (on the CPU) and check
that the pins catch every one of them.  Each mutant runs in a child process, so a
mutant that reads out of bounds and crashes also counts as caught."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "dropped_scale": ("score[j] = softmax_scale * dot;", "score[j] = dot;"),
    "gqa_modulo": ("hk = h / group;", "hk = h % num_heads_k;"),
    "left_window_sign": ("j < i + c - wl", "j < i + c + wl"),
    "top_left_alignment": ("int64_t c = sk - sq;", "int64_t c = 0;"),
    "right_window_dropped": ("if (wr >= 0 && j > i + c + wr) return 0;", ""),
    "page_slot_swapped": ("block * s[0] + (j % page_block_size) * s[1]",
                          "block * s[1] + (j % page_block_size) * s[0]"),
    "page_index_modulo": ("block_table[b * bt_row_stride + j / page_block_size]",
                          "block_table[b * bt_row_stride + j % page_block_size]"),
    "values_from_keys": ("kv_row(v, kv_stride", "kv_row(k, kv_stride"),
    "lse_without_max": ("lse[r] = m + log(l);", "lse[r] = log(l);"),
    "f16_exponent_bias": ("expo - 25", "expo - 24"),
    "no_normalisation": ("o[d] /= l;", "o[d] /= 1.0;"),
    "exp_without_max": ("double w = exp(score[j] - m);", "double w = exp(score[j]);"),
    "empty_row_lse_zero": ("lse[r] = -INFINITY;", "lse[r] = 0.0;"),
    "alibi_sign": ("return -slope * fabs(", "return slope * fabs("),
    "alibi_no_abs": ("fabs((double)(i + c - j))", "((double)(i + c - j))"),
    "alibi_top_left": ("fabs((double)(i + c - j))", "fabs((double)(i - j))"),
    "alibi_kv_head": ("alibi_slopes[h]", "alibi_slopes[hk]"),
}


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = """
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import _pins
lib = oracle.load({so!r})
attn = lambda *a, **kw: oracle.attention(*a, lib=lib, **kw)
try:
    for pin in _pins.ALL_PINS:
        pin(attn)
    _pins.pin_decoders(lambda dt, b: oracle.decode(dt, b, lib=lib))
except AssertionError:
    sys.exit(3)
sys.exit(0)
"""


def _pins_pass(so):
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, so=so)],
                       capture_output=True, timeout=600)
    return r.returncode == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "libm.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", c, "-o", so, "-lm"],
                       check=True, capture_output=True)
        assert not _pins_pass(so), f"mutant {name} passed every pin"


def test_unmutated_source_passes_in_child():
    """The child harness itself passes on the committed source (so a failure above is the
    mutation's doing)."""
    with tempfile.TemporaryDirectory() as d:
        so = os.path.join(d, "libo.so")
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", SRC, "-o", so, "-lm"],
                       check=True, capture_output=True)
        assert _pins_pass(so)
