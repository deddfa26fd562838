"""Failure detection on the GPU without a fault: the test hook leaves one ring
slot of one CTA unfilled, so that CTA's bounded pipeline waits run out
(about a second each). The call must report DA_DEVERR_TIMEOUT, publish NaN
for the affected group only, and leave the context usable: the next call on
the same stream, with the workspace zeroed again, is correct."""
import pytest
import torch

import decode_attention_static_gb300 as da
import workloads as W
from gpu_helpers import assert_close, oracle_step

pytestmark = pytest.mark.gpu

DA_DEVERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()


def _run(step, hint, ws):
    d = step.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids, workspace=ws,
                             max_kv_len_hint=hint, err_flag=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("case", ["flat", "cluster"])
def test_pipeline_timeout_is_reported_and_the_context_survives(ora, case):
    if case == "flat":
        step, hint = W.long_context(seed=40), 32768        # flat split plan, merge through the workspace
    else:
        step, hint = W.mha_sweep(4096, seed=41), 4096      # one cluster per head, on-chip merge
    G = step.n_head // step.n_kv_head
    ws = da.alloc_workspace(step.B, step.n_head, step.n_kv_head, step.head_dim, step.capacity)
    da.test_skip_slot(1)
    try:
        out, err = _run(step, hint, ws)
    finally:
        da.test_skip_slot(-1)
    assert err & DA_DEVERR_TIMEOUT, f"error flag {err}"
    o = out.float()
    assert bool(torch.isnan(o[0, :G]).all()), "the timed-out group must be NaN"
    assert bool(torch.isfinite(o[0, G:]).all()), "other groups must be unaffected"
    _, _, ref = oracle_step(ora, step)
    assert_close(out[:, G:], ref[:, G:], f"{case}: unaffected groups")
    # the same context, the workspace zeroed again: a normal call is correct
    da.workspace_init(ws)
    out2, err2 = _run(step, hint, ws)
    assert err2 == 0
    assert_close(out2, ref, f"{case}: after the timeout")
