"""decode_attn_fwd_static_scratch: the entry point for callers that may not
allocate GPU memory (for instance a plugin that only gets input and output
buffers from the server or audio engine hosting it). Its split partials live
in the library's own fixed device array instead of a caller workspace.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

import decode_attention_static_gb300 as da
from decode_attention_static_gb300 import workloads as W
from gpu_helpers import assert_close, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()


def _scratch_need(step, hint):
    s, cs = da.splits_for(step.B, step.n_head, step.n_kv_head, step.head_dim, step.capacity, hint,
                          W.torch_dtype(step.dtype))
    # several clusters per group: a 4 KiB region of arrival counters, then
    # fp32 per-cluster partials [B, n_head, S / cluster, D + 2]
    nc = s // cs
    return s, (4096 + step.B * step.n_head * nc * (step.head_dim + 2) * 4 if nc > 1 else 0)


def test_matches_workspace_entry_point_on_two_calls_in_a_row(ora):
    """Two different decode steps back to back through the no-allocation entry
    point: each matches decode_attn_fwd (with a caller workspace) and the
    fp64 oracle, so the second call does not see the first call's partials."""
    steps = [W.long_context(seed=21, kv_len=30001), W.long_context(seed=22, kv_len=20000)]
    for step in steps:
        splits, need = _scratch_need(step, 0)
        assert splits > 1 and 0 < need <= da.STATIC_SCRATCH_BYTES  # the scratch path is exercised
    outs = []
    for step in steps:
        d = step.to("cuda")
        da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = da.decode_attn_fwd_static_scratch(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), err_flag=err)
        ref = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous())
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref.double().cpu().numpy(), "static scratch vs workspace entry point")
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        outs.append((step, got.clone()))
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
        splits, need = _scratch_need(step, 0)
        if need > da.STATIC_SCRATCH_BYTES:
            break
    else:
        pytest.skip(f"no candidate split plan exceeds the scratch array on this GPU (largest {need} B)")
    d = step.to("cuda")
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_fwd_static_scratch(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous())
    assert e.value.status == -2
    # nothing was enqueued and the array is untouched: a fitting call still works
    small = W.long_context(seed=25, kv_len=20000)
    ds = small.to("cuda")
    da.kvcache_append(ds.k_cache, ds.v_cache, ds.k_new, ds.v_new, ds.position_ids)
    got = da.decode_attn_fwd_static_scratch(ds.q, ds.k_cache, ds.v_cache, ds.kv_len.contiguous())
    ref = da.decode_attn_fwd(ds.q, ds.k_cache, ds.v_cache, ds.kv_len.contiguous())
    torch.cuda.synchronize()
    assert bool(torch.isfinite(got.float()).all())
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
