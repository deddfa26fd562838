"""Plant plausible mistakes in copies of the oracle source and check that the
pin suite catches every one of them (CPU only; the shipped oracle is never
modified). Each mutant runs in its own process so that a crash also counts
as caught."""
import json
import pathlib
import subprocess
import sys

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
SOURCE = (ROOT / "oracle" / "oracle.c").read_text()

# (name, original text, mutated text)
MUTANTS = [
    ("head map h % n_kv_head", "const int g = h / G;", "const int g = h % n_kv_head;"),
    ("exp sign flipped", "x[j] = exp(x[j] - m);", "x[j] = exp(m - x[j]);"),
    ("max not subtracted", "x[j] = exp(x[j] - m);", "x[j] = exp(x[j]);"),
    ("scale dropped", "x[j] = scale * dot;", "x[j] = dot;"),
    ("normalisation dropped", "o[d] = acc / Z;", "o[d] = acc;"),
    ("K used for V", "acc += x[j] * decode(V[", "acc += x[j] * decode(K["),
    ("V read one row past the prefix", "for (int j = 0; j < L; ++j) acc +=",
     "for (int j = 0; j <= L && j < capacity; ++j) acc +="),
    ("q head ignored", "const uint16_t* qr = q + bh * head_dim;",
     "const uint16_t* qr = q + (int64_t)b * n_head * head_dim;"),
    ("K operand transposed", "decode(K[(int64_t)j * head_dim + d], dtype)",
     "decode(K[(int64_t)(d % L) * head_dim + (j % head_dim)], dtype)"),
    ("max over all but the last row", "for (int j = 1; j < L; ++j)\n      if (x[j] > m) m = x[j];",
     "for (int j = 1; j < L - 1; ++j)\n      if (x[j] > m) m = x[j];"),
    ("fp16 exponent bias off by one", "expo - 25", "expo - 24"),
    ("fp16 subnormal scale", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("bf16 exponent field misplaced", "int expo = (h >> 7) & 0xff;", "int expo = (h >> 8) & 0xff;"),
    ("append row off by one", "* capacity + p) * head_dim;", "* capacity + (p + 1) % capacity) * head_dim;"),
    ("append ignores V", "memcpy(v_cache + dst, v_new + src", "memcpy(v_cache + dst, k_new + src"),
    ("kv_len bound not checked", "if (L < 1 || L > capacity) {", "if (L < 1) {"),
    ("position bound not checked", "if (p < 0 || p >= capacity) {", "if (p < 0) {"),
    ("rope partner sign flipped", "r = a - bb;", "r = a + bb;"),
    ("rope partner index", "decode(xr[d + half], dtype); /* rotate_half", "decode(xr[d], dtype); /* rotate_half"),
    ("rope sin replaced by cos", "const float bb = yv * s[d];\n          r = a - bb;",
     "const float bb = yv * c[d];\n          r = a - bb;"),
    ("rope table row ignored", "const float* c = cos_table + (int64_t)p * head_dim;",
     "const float* c = cos_table;"),
    ("rope position bound not checked", "if (p < 0 || p >= rows) {", "if (p < 0) {"),
    ("f16 encoder truncates", "if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;", ""),
    ("f16 encoder subnormal shift", "const int shift = -e - 1;", "const int shift = -e;"),
    ("bf16 encoder ties away from zero", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
]


def _mutant_lib(tmp_path, name, old, new):
    assert SOURCE.count(old) >= 1, f"mutation anchor for '{name}' not found in oracle.c"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(SOURCE.replace(old, new))
    sys.path.insert(0, str(ROOT))
    from oracle import build

    return build.compile_oracle(src, tmp_path / "liboracle_mutant.so", openmp=False)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    lib = _mutant_lib(tmp_path, name, old, new)
    r = subprocess.run([sys.executable, str(ROOT / "tests" / "oracle_pins.py"), str(lib)],
                       capture_output=True, text=True, cwd=str(ROOT), timeout=300,
                       env={"PYTHONPATH": f"{ROOT}:{ROOT / 'tests'}", "PATH": "/usr/bin:/bin"})
    if r.returncode != 0:
        return  # the mutant crashed the pin run: caught
    results = json.loads(r.stdout.strip().splitlines()[-1])
    failed = [k for k, v in results.items() if v != "ok"]
    assert failed, f"mutant '{name}' passed every pin"
