"""decode_attn_fwd_static_scratch: the entry point for callers that may not
allocate GPU memory (for instance a plugin that only gets input and output
buffers from the server or audio engine hosting it). Its split partials live
in the library's own fixed device array instead of a caller workspace; every
call zero-fills its own arrival counters there first, so nothing an earlier
call left behind (a smaller or larger plan, a timed-out pipeline, two calls
that overlapped) can spoil the next ordered call.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

import decode_attention_static_gb300 as da
import workloads as W
from gpu_helpers import assert_close, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()


def _scratch_need(step, hint=0):
    s, cs = da.splits_for(step.B, step.n_head, step.n_kv_head, step.head_dim, step.capacity, hint,
                          W.torch_dtype(step.dtype))
    # several clusters per group: a 4 KiB region of arrival counters, then
    # fp32 per-cluster partials [B, n_head, S / cluster, D + 2]
    nc = s // cs
    return s, (4096 + step.B * step.n_head * nc * (step.head_dim + 2) * 4 if nc > 1 else 0)


def _appended(step):
    d = step.to("cuda")
    da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    return d


def _check_against_workspace_entry(d, what):
    """One static-scratch call: no device error, bit-equal to decode_attn_fwd
    with a caller workspace. Returns the output."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = da.decode_attn_fwd_static_scratch(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), err_flag=err)
    ref = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous())
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error flag {int(err.item())}"
    assert_close(got, ref.double().cpu().numpy(), f"{what}: static scratch vs workspace entry point")
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"{what}: not bit-equal"
    return got


def test_matches_workspace_entry_point_on_two_calls_in_a_row(ora):
    """Two decode calls back to back through the no-allocation entry point,
    the second with a smaller split plan than the first (so the array still
    holds the first call's larger set of partials): each matches
    decode_attn_fwd with a caller workspace bit for bit, and the fp64 oracle
    within tolerance."""
    first = W.decode_step(2, 32, 8, 128, 32768, "bf16", [30000, 25000], seed=21)
    second = W.decode_step(1, 16, 4, 128, 32768, "bf16", [20000], seed=22)
    needs = [_scratch_need(s)[1] for s in (first, second)]
    assert all(0 < n <= da.STATIC_SCRATCH_BYTES for n in needs), needs  # the scratch path is exercised
    assert needs[1] < needs[0]
    outs = [(s, _check_against_workspace_entry(_appended(s), f"call {i}").clone()) for i, s in
            enumerate((first, second))]
    for step, got in outs:
        _, _, oref = oracle_step(ora, step)
        assert_close(got, oref, "static scratch vs oracle")


def test_rejects_sizes_beyond_the_scratch_limit():
    """A split plan needing more than the fixed array is refused before any
    launch (DA_ERR_SHAPE). Two sequences of a long cache with 8 query heads
    per KV head give a flat plan of about 1.2 MiB of partials on a 152-SM
    GPU; the first candidate shape whose plan exceeds the array is used."""
    candidates = [W.decode_step(2, 64, 8, 128, 32768, "bf16", [32767, 30000], seed=23),
                  W.decode_step(2, 32, 8, 128, 32768, "bf16", [32767, 32767], seed=24)]
    for step in candidates:
        splits, need = _scratch_need(step)
        if need > da.STATIC_SCRATCH_BYTES:
            break
    else:
        pytest.skip(f"no candidate split plan exceeds the scratch array on this GPU (largest {need} B)")
    d = step.to("cuda")
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_fwd_static_scratch(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous())
    assert e.value.status == -2
    # nothing was enqueued: a fitting call still works
    _check_against_workspace_entry(_appended(W.long_context(seed=25, kv_len=20000)), "after a rejection")


def test_timed_out_call_is_reported_and_the_next_call_is_correct(ora):
    """The failure-detection hook leaves one ring slot of one CTA of a
    static-scratch call unfilled: its bounded waits run out (about a second
    each), the call reports DA_DEVERR_TIMEOUT and NaN rows for that KV head's
    query heads only. The very next static-scratch call, with nothing reset
    by the caller, is bit-equal to decode_attn_fwd and matches the oracle."""
    step = W.long_context(seed=26, kv_len=30001)
    assert _scratch_need(step)[1] > 0  # a flat plan: partials go through the array
    G = step.n_head // step.n_kv_head
    d = _appended(step)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da.test_skip_slot(1)
    try:
        bad = da.decode_attn_fwd_static_scratch(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), err_flag=err)
        torch.cuda.synchronize()
    finally:
        da.test_skip_slot(-1)
    assert int(err.item()) & da.DA_DEVERR_TIMEOUT, f"error flag {int(err.item())}"
    assert bool(torch.isnan(bad[0, :G].float()).all()), "the timed-out group must be NaN"
    assert bool(torch.isfinite(bad[0, G:].float()).all()), "other groups must be unaffected"
    got = _check_against_workspace_entry(d, "after the time-out")
    _, _, ref = oracle_step(ora, step)
    assert_close(got, ref, "after the time-out vs oracle")


def test_overlapping_calls_leave_nothing_to_reset(ora):
    """Two static-scratch calls of different shapes launched on two streams
    without ordering race on the shared array (their results are not
    checked). Once both have finished, an ordered call is correct again with
    nothing reset by the caller."""
    a = _appended(W.decode_step(2, 32, 8, 128, 32768, "bf16", [30000, 28000], seed=27))
    step_b = W.long_context(seed=28, kv_len=24000)
    b = _appended(step_b)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(4):
        with torch.cuda.stream(s1):
            da.decode_attn_fwd_static_scratch(a.q, a.k_cache, a.v_cache, a.kv_len.contiguous())
        with torch.cuda.stream(s2):
            da.decode_attn_fwd_static_scratch(b.q, b.k_cache, b.v_cache, b.kv_len.contiguous())
    torch.cuda.synchronize()
    got = _check_against_workspace_entry(b, "after overlapping calls")
    _, _, ref = oracle_step(ora, step_b)
    assert_close(got, ref, "after overlapping calls vs oracle")
