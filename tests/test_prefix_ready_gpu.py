"""The ordering promise (da_set_prefix_ready): with it, a single-sequence call
with a length bound copies its first tiles before waiting for the previous
kernel on the stream. Where the promise holds the results must be those of
the default ordering bit for bit (the same tiles, the same arithmetic) and
match the oracle: early tiles kept (bound == length) and discarded (bound !=
length), every split plan, the rotary step, the layers call, graph capture,
and the time-out hook on a slot issued before the wait."""
import numpy as np
import pytest
import torch

import decode_attention_static_gb300 as da
import workloads as W
from gpu_helpers import assert_close, bits, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()
    yield
    da.set_prefix_ready(False)


def _fused(step: W.DecodeStep, hint: int, ready: bool):
    d = step.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da.set_prefix_ready(ready)
    try:
        out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids,
                                 max_kv_len_hint=hint, err_flag=err)
    finally:
        da.set_prefix_ready(False)
    torch.cuda.synchronize()
    return d, out, int(err.item())


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


CASES = {
    "mha_kv1024_cluster": lambda: W.mha_sweep(1024, seed=70),
    "mha_kv4096_cluster": lambda: W.mha_sweep(4096, seed=71),
    "mha_kv8192_cluster": lambda: W.mha_sweep(8192, seed=72),
    "gqa_kv32768_flat": lambda: W.long_context(seed=73),
    "gqa_ragged_tail": lambda: W.long_context(seed=74, kv_len=20001, capacity=20480),
    "tiny_gqa": lambda: W.tiny_gqa(seed=75),
    "d64_g8": lambda: W.decode_step(1, 8, 1, 64, 3000, "bf16", [2999], seed=76),
}


@pytest.mark.parametrize("name", list(CASES))
def test_kept_early_tiles_match_default_ordering_and_oracle(ora, name):
    step = CASES[name]()
    L = int(step.kv_len[0])
    kb, vb, ref = oracle_step(ora, step)
    d0, out0, err0 = _fused(step, L, ready=False)
    d1, out1, err1 = _fused(step, L, ready=True)
    assert err0 == 0 and err1 == 0
    assert _same(out1, out0), f"{name}: output differs from the default ordering"
    assert np.array_equal(bits(d1.k_cache), kb) and np.array_equal(bits(d1.v_cache), vb)
    assert_close(out1, ref, name)


@pytest.mark.parametrize("L,delta", [(1024, -700), (1024, -1), (1024, 1), (1024, 64), (1024, 900),
                                     (4096, -1), (4096, 900)])
def test_discarded_early_tiles(ora, L, delta):
    """Bound off the length: the early tiles (copied before the wait when the
    bound's chunks are short) are discarded and the call is still exact."""
    step = W.decode_step(1, 16, 16, 128, 6000, "f16", [L - 1], seed=77)
    hint = L + delta
    kb, vb, ref = oracle_step(ora, step)
    _, out0, _ = _fused(step, hint, ready=False)
    d1, out1, err1 = _fused(step, hint, ready=True)
    assert err1 == 0
    assert _same(out1, out0)
    assert np.array_equal(bits(d1.k_cache), kb) and np.array_equal(bits(d1.v_cache), vb)
    assert_close(out1, ref, f"bound {hint}")


def test_attention_call_with_ready_prefix(ora):
    """decode_attn_fwd reads rows [0, bound) before the wait: the append is
    finished (synchronised) before the call, so the promise holds."""
    step = W.mha_sweep(1024, seed=78)
    kb, vb, ref = oracle_step(ora, step)
    d = step.to("cuda")
    da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    torch.cuda.synchronize()
    lens = d.kv_len.contiguous()
    out0 = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, lens, max_kv_len_hint=1024)
    with da.prefix_ready():
        out1 = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, lens, max_kv_len_hint=1024)
    torch.cuda.synchronize()
    assert _same(out1, out0)
    assert_close(out1, ref, "attention call")


@pytest.mark.parametrize("kv", [1024, 4096])
def test_rotary_step_with_ready_prefix(ora, kv):
    step = W.decode_step(1, 16, 16, 128, kv, "f16", [kv - 1], seed=79 + kv)
    cos, sin = W.random_rope_tables(kv, 128, seed=kv)
    outs = []
    for ready in (False, True):
        d = step.to("cuda")
        da.set_prefix_ready(ready)
        try:
            out = da.decode_step_rope_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, cos.cuda(), sin.cuda(),
                                          d.position_ids, max_kv_len_hint=kv)
        finally:
            da.set_prefix_ready(False)
        torch.cuda.synchronize()
        outs.append((d, out))
    (d0, o0), (d1, o1) = outs
    assert _same(o1, o0)
    assert _same(d1.k_cache, d0.k_cache) and _same(d1.v_cache, d0.v_cache)


def test_graph_of_layers_with_ready_prefix(ora):
    """A CUDA graph of per-layer fused calls on separate layer caches (the
    promise holds: consecutive kernels touch different caches), replayed:
    the same outputs and caches as the default ordering, and the oracle's."""
    layers, kv = 6, 2048
    steps = [W.mha_sweep(kv, seed=90 + l) for l in range(layers)]

    def run(ready: bool):
        dev = [s.to("cuda") for s in steps]
        out = [torch.empty_like(d.q) for d in dev]
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        da.set_prefix_ready(ready)
        try:
            with torch.cuda.graph(g):
                for l, d in enumerate(dev):
                    da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids, out=out[l],
                                       max_kv_len_hint=kv)
        finally:
            da.set_prefix_ready(False)
        g.replay()
        torch.cuda.synchronize()
        return dev, out

    d0, o0 = run(False)
    d1, o1 = run(True)
    for l in range(layers):
        assert _same(o1[l], o0[l]), f"layer {l}"
        assert _same(d1[l].k_cache, d0[l].k_cache)
    for l in (0, layers - 1):
        kb, vb, ref = oracle_step(ora, steps[l])
        assert np.array_equal(bits(d1[l].k_cache), kb)
        assert_close(o1[l], ref, f"layer {l}")


def test_layers_call_with_ready_prefix():
    layers, kv = 4, 1024
    steps = [W.mha_sweep(kv, seed=100 + l) for l in range(layers)]
    stack = lambda name: torch.stack([getattr(s, name) for s in steps]).cuda()  # noqa: E731
    res = []
    for ready in (False, True):
        q, kc, vc, kn, vn = (stack(n) for n in ("q", "k_cache", "v_cache", "k_new", "v_new"))
        p = steps[0].position_ids.cuda()
        da.set_prefix_ready(ready)
        try:
            out = da.decode_step_layers_fwd(q, kc, vc, kn, vn, p, max_kv_len_hint=kv)
        finally:
            da.set_prefix_ready(False)
        torch.cuda.synchronize()
        res.append((out, kc))
    assert _same(res[1][0], res[0][0]) and _same(res[1][1], res[0][1])


@pytest.mark.parametrize("slot", [0, 1])
def test_timeout_on_a_slot_issued_before_the_wait(ora, slot):
    """The test hook leaves an early slot (normally copied before the wait)
    unfilled: the call reports DA_DEVERR_TIMEOUT, NaN for that group only,
    and the next call on the same context is correct. (kv 1024: two-tile
    chunks, both early slots copied before the wait.)"""
    step = W.mha_sweep(1024, seed=110)
    G = step.n_head // step.n_kv_head
    ws = da.alloc_workspace(1, step.n_head, step.n_kv_head, step.head_dim, step.capacity)
    d = step.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da.test_skip_slot(slot)
    da.set_prefix_ready(True)
    try:
        out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids, workspace=ws,
                                 max_kv_len_hint=1024, err_flag=err)
        torch.cuda.synchronize()
    finally:
        da.test_skip_slot(-1)
        da.set_prefix_ready(False)
    assert int(err.item()) & da.DA_DEVERR_TIMEOUT
    o = out.float()
    assert bool(torch.isnan(o[0, :G]).all())
    assert bool(torch.isfinite(o[0, G:]).all())
    _, _, ref = oracle_step(ora, step)
    assert_close(out[:, G:], ref[:, G:], "unaffected groups")
    da.workspace_init(ws)
    _, out2, err2 = _fused(step, 1024, ready=True)
    assert err2 == 0
    assert_close(out2, ref, "after the timeout")


@pytest.mark.parametrize("hint_delta", [0, -100, 37])
def test_rotary_step_d64_with_ready_prefix(ora, hint_delta):
    """Rotary step at head_dim 64, 8 query / 2 KV heads, with the bound on and
    off the length (the rotated slot issued after the wait, kept or dropped)."""
    cap, pos = 2000, 1499
    step = W.decode_step(1, 8, 2, 64, cap, "bf16", [pos], seed=120)
    cos, sin = W.random_rope_tables(cap, 64, seed=121)
    outs = []
    for ready in (False, True):
        d = step.to("cuda")
        da.set_prefix_ready(ready)
        try:
            out = da.decode_step_rope_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, cos.cuda(), sin.cuda(),
                                          d.position_ids, max_kv_len_hint=pos + 1 + hint_delta)
        finally:
            da.set_prefix_ready(False)
        torch.cuda.synchronize()
        outs.append((d, out))
    (d0, o0), (d1, o1) = outs
    assert _same(o1, o0)
    assert _same(d1.k_cache, d0.k_cache) and _same(d1.v_cache, d0.v_cache)


def test_batch_is_unaffected_by_the_promise(ora):
    """The promise only changes single-sequence calls with a bound: a batch
    gives the same bits either way."""
    step = W.batched_streaming(seed=5)
    hint = int(step.position_ids.max()) + 1
    r0 = _fused(step, hint, ready=False)
    r1 = _fused(step, hint, ready=True)
    assert r0[2] == 0 and r1[2] == 0
    assert _same(r1[1], r0[1])
