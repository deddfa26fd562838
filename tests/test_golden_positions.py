"""The position -> active-length mapping against the numbers the pages print
(tests/golden/kv_len_from_position.json), through the synthetic-input
generator that feeds both the oracle and the CUDA path (CPU only)."""
import json
import pathlib

import workloads as W

GOLD = json.loads((pathlib.Path(__file__).parent / "golden" / "kv_len_from_position.json").read_text())


def test_patched_rows_attended():
    for case in GOLD["cases"]:
        step = W.decode_step(1, 2, 1, 8, case["capacity"], "f16", [case["position_id"]], seed=0)
        assert int(step.kv_len[0]) == case["rows_attended_patched"], case["cite"]
        assert step.capacity == case["rows_attended_baseline"], case["cite"]
        # the generator leaves exactly the rows before position_id filled; the
        # append fills row position_id, after which kv_len rows are finite
        finite_rows = int(step.k_cache[0, 0].float().isfinite().all(dim=-1).sum())
        assert finite_rows == case["position_id"]


def test_generation_lengths():
    g = GOLD["generation"]
    gen = W.s2pro_generation(layers=1, steps=3)
    assert gen.prompt == g["prompt_T"] == g["prefill_kv_len"]
    assert gen.capacity == g["capacity"]
    assert gen.position(0) + 1 == g["first_decode_kv_len"]
    lo = 100.0 * g["prompt_T"] / g["capacity"]
    hi = 100.0 * g["context_end"] / g["capacity"]
    assert round(lo, 1) == g["active_fraction_low_pct"]
    assert abs(hi - g["active_fraction_high_pct"]) < 0.1
