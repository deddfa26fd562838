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


@pytest.mark.parametrize("case", ["flat", "cluster", "gqa_cluster"])
def test_pipeline_timeout_is_reported_and_the_context_survives(ora, case):
    if case == "flat":
        # flat split plan, merge through the workspace; tensor-core scores
        step, hint = W.long_context(seed=40), 32768
    elif case == "cluster":
        step, hint = W.mha_sweep(4096, seed=41), 4096      # one cluster per head, on-chip merge
    else:
        # four heads per KV head, one cluster per group, CUDA-core scores
        step, hint = W.long_context(seed=42, kv_len=2048, capacity=2048), 2048
        assert da.kernel_for(1, step.n_head, step.n_kv_head, step.head_dim, 2048, 2048, step.q.dtype) == "cuda_cores"
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


def test_layers_call_timeout_is_reported_and_the_context_survives(ora):
    """The same time-out inside the one-launch layers call: the hook leaves a
    ring slot of layer 0's first KV head unfilled, so only that layer's query
    heads of that KV head become NaN; every other layer and head is correct,
    and the next layers call on the same workspace (zeroed again) is correct
    everywhere."""
    layers, B, H, Hkv, D, cap = 4, 1, 32, 8, 128, 1024
    steps = [W.decode_step(B, H, Hkv, D, cap, "bf16", [634], seed=90 + l) for l in range(layers)]
    G = H // Hkv
    stack = lambda name: torch.stack([getattr(s, name) for s in steps]).cuda()  # noqa: E731

    def run():
        q, kc, vc, kn, vn = (stack(n) for n in ("q", "k_cache", "v_cache", "k_new", "v_new"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = da.decode_step_layers_fwd(q, kc, vc, kn, vn, steps[0].position_ids.cuda(), workspace=ws,
                                        max_kv_len_hint=635, err_flag=err)
        torch.cuda.synchronize()
        return out, int(err.item())

    ws = da.alloc_workspace(layers * B, H, Hkv, D, cap)
    da.test_skip_slot(1)
    try:
        out, err = run()
    finally:
        da.test_skip_slot(-1)
    assert err & DA_DEVERR_TIMEOUT, f"error flag {err}"
    o = out.float()
    assert bool(torch.isnan(o[0, 0, :G]).all()), "the timed-out group must be NaN"
    assert bool(torch.isfinite(o[0, 0, G:]).all()) and bool(torch.isfinite(o[1:]).all()), "others unaffected"
    refs = [oracle_step(ora, s)[2] for s in steps]
    assert_close(out[0, :, G:], refs[0][:, G:], "layer 0, unaffected heads")
    for l in range(1, layers):
        assert_close(out[l], refs[l], f"layer {l}")
    da.workspace_init(ws)
    out2, err2 = run()
    assert err2 == 0
    for l in range(layers):
        assert_close(out2[l], refs[l], f"layer {l} after the time-out")
