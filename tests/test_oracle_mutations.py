"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins catch each one.  The copy lives in a temporary directory; the real
oracle is never modified."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("rope rotation direction", "a * c - b * s, b * c + a * s", "a * c + b * s, b * c - a * s"),
    ("gqa head mapping", "g = h // n_rep", "g = h % nkv"),
    ("attention scale", "scale = 1.0 / np.sqrt(F64(d))", "scale = 1.0 / F64(d)"),
    ("rope exponent", "-2.0 * i / d", "-1.0 * i / d"),
    ("qk norm dropped", 'q = rms_norm(q, W["q_norm"], eps)', "q = q"),
    ("kv written after attention", "S = int(pos[-1]) + 1", "S = int(pos[0])"),
    ("silu on up", "linear(silu(linear(xn, W_gate)) * linear(xn, W_up), W_down)",
     "linear(linear(xn, W_gate) * silu(linear(xn, W_up)), W_down)"),
    ("rms without mean", "ms = np.mean(x * x, axis=-1, keepdims=True)",
     "ms = np.sum(x * x, axis=-1, keepdims=True)"),
    ("causal mask off by one", "visible = np.arange(S)[None, :] <= _f64(q_pos)[:, None]",
     "visible = np.arange(S)[None, :] < _f64(q_pos)[:, None] + 2"),
    ("residual dropped", 'x = x + linear(o.reshape(T, nq * d), W["o"])',
     'x = linear(o.reshape(T, nq * d), W["o"])'),
    ("argmax picks last tie", "np.flatnonzero(v == np.max(v))[0]", "np.flatnonzero(v == np.max(v))[-1]"),
    ("transposed weight", "return _f64(x) @ _f64(W).T", "return _f64(x) @ _f64(W).reshape(_f64(W).shape[::-1])"),
    ("budget slack dropped", "want = 2 * n_audio + 128", "want = 2 * n_audio"),
    ("budget floor ignored", "min(max(want, floor_new), ceiling - T_prompt)", "min(want, ceiling - T_prompt)"),
    ("budget cap ignored", "min(max(want, floor_new), ceiling - T_prompt)", "max(want, floor_new)"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    for d in ("oracle", "tests", "speech_decoder_gb300"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc", "golden"))
    src = (tmp_path / "oracle" / "decoder.py").read_text()
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    (tmp_path / "oracle" / "decoder.py").write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin:\n{r.stdout[-2000:]}"


E4M3_MUTATIONS = [
    ("e4m3 ties away from zero", "np.round(a / step) * step", "np.floor(a / step + 0.5) * step"),
    ("e4m3 subnormal spacing", "e = np.maximum(ex - 1, -6)", "e = np.maximum(ex - 1, -7)"),
    ("e4m3 two mantissa bits", "step = np.ldexp(1.0, e - 3)", "step = np.ldexp(1.0, e - 2)"),
    ("e4m3 no saturation", "q = np.minimum(np.round(a / step) * step, E4M3_MAX)", "q = np.round(a / step) * step"),
    ("row scale not the smallest", "e = np.where(f == np.float32(0.5), x - 1, x)", "e = x"),
    ("e4m3 exponent bias", "(1.0 + m / 8.0) * np.ldexp(1.0, e - 7)", "(1.0 + m / 8.0) * np.ldexp(1.0, e - 8)"),
]


@pytest.mark.parametrize("name,old,new", E4M3_MUTATIONS, ids=[m[0] for m in E4M3_MUTATIONS])
def test_e4m3_pins_catch_planted_mistake(tmp_path, name, old, new):
    for d in ("oracle", "tests"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("__pycache__", "golden"))
    src = (tmp_path / "oracle" / "e4m3.py").read_text()
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    (tmp_path / "oracle" / "e4m3.py").write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_e4m3_pins.py"], cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin:\n{r.stdout[-2000:]}"
    assert " failed" in r.stdout, f"the pins did not run:\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
