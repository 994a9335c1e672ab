"""The pins are strong enough: each plausible mistake planted in a copy of the C
oracle (a dropped term, a wrong sign, a wrong index, a transposed operand, a
swapped operand, a reversed order) makes the pin suite fail.

Each case compiles the mutated copy into a temporary directory and runs
tests/test_oracle_pins.py against it in a child process (the oracle module is
pointed at the copy before any test imports it).  A control run of the
unmodified copy must pass, so a failure really comes from the planted mistake.
The mutations keep every memory access in bounds.  CPU only; no GPU is
touched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, original text, planted text, occurrences replaced)
MUTATIONS = [
    ("router weights not renormalised over the kept experts",
     "  for (int j = 0; j < k; ++j) w[j] = p[idx[j]] / s;",
     "  for (int j = 0; j < k; ++j) w[j] = p[idx[j]];", 1),
    ("top-k ties go to the higher expert index",
     "return la > lb || (la == lb && a < b); }",
     "return la > lb || (la == lb && a > b); }", 1),
    ("tokens placed in descending order inside an expert",
     "      int32_t row = offsets[e] + fill[e]++;",
     "      int32_t row = offsets[e + 1] - 1 - fill[e]++;", 1),
    ("gate and up swapped in SwiGLU",
     "  for (int i = 0; i < I; ++i) a[i] = silu(g[i]) * u[i];",
     "  for (int i = 0; i < I; ++i) a[i] = silu(u[i]) * g[i];", 2),
    ("W_gate read transposed",
     "      g[i] += xv * bf(wg[(int64_t)h * I + i]);",
     "      g[i] += xv * bf(wg[(int64_t)i * H + h]);", 1),
    ("dSwiGLU derivative term dropped from dG",
     "        dg[i] = da[i] * ui * sg * (1.0 + gi * (1.0 - sg));",
     "        dg[i] = da[i] * ui * sg;", 1),
    ("router weight left out of dA",
     "        for (int h = 0; h < H; ++h) dyw[h] = w * bf(dyt[h]);",
     "        for (int h = 0; h < H; ++h) dyw[h] = bf(dyt[h]);", 1),
    ("d_logits with the wrong sign",
     "    for (int j = 0; j < k; ++j) dp[sel[j]] = (gd[j] - gbar) / P;",
     "    for (int j = 0; j < k; ++j) dp[sel[j]] = (gbar - gd[j]) / P;", 1),
    ("dx misses the up branch",
     "          for (int i = 0; i < I; ++i) acc += dg[i] * bf(wg[i]) + du[i] * bf(wu[i]);",
     "          for (int i = 0; i < I; ++i) acc += dg[i] * bf(wg[i]);", 1),
    ("MXFP8 scale one power of two too small (blocks saturate)",
     "  if (amax > ldexp(448.0, X)) X += 1;",
     "", 1),
]

_BOOT = """
import sys
sys.path.insert(0, {root!r})
from oracle import oracle as O
O._SRC, O._OUT_DIR, O._LIB = {src!r}, {out!r}, {lib!r}
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", {pins!r}]))
"""


def _run_pins(tmp_path, source):
    src = tmp_path / "moe_oracle.c"
    src.write_text(source)
    boot = _BOOT.format(root=ROOT, src=str(src), out=str(tmp_path), lib=str(tmp_path / "libmoe_oracle.so"),
                        pins=PINS)
    r = subprocess.run([sys.executable, "-c", boot], cwd=ROOT, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def test_control_copy_passes(tmp_path):
    code, out = _run_pins(tmp_path, open(SRC).read())
    assert code == 0, out


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, count):
    source = open(SRC).read()
    assert source.count(old) == count, f"mutation target not found as expected: {old!r}"
    code, out = _run_pins(tmp_path, source.replace(old, new))
    assert code != 0, f"no pin caught: {name}\n{out}"
    assert "failed" in out or "Error" in out, out
