"""GPU parity: the CUDA library through its C ABI against the fp64 oracle on
the seeded synthetic workloads, at full size, plus edge cases. Tolerances:
rel-Frobenius <= 5e-3 and max-abs <= 2e-2 for the attention output; the
cache append is compared bit for bit, NaN tail included."""
import ctypes

import numpy as np
import pytest
import torch

import decode_attention_static_gb300 as da
import workloads as W
from gpu_helpers import THREADS, assert_close, bits, check_step, gpu_step, oracle_step

pytestmark = pytest.mark.gpu

FUSED = [False, True]
FUSED_IDS = ["append+attend", "fused_step"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_tiny_gqa(ora, fused):
    check_step(ora, W.tiny_gqa(seed=0), fused, what="tiny GQA")


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("kv_len", W.MHA_SWEEP_KV_LENS)
def test_mha_sweep(ora, kv_len, fused):
    check_step(ora, W.mha_sweep(kv_len, seed=1), fused, what=f"MHA kv {kv_len}")


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("kv_len", [2048, 3072, 5000, 6144])
def test_mha_mid_lengths(ora, kv_len, fused):
    """Prefixes between the sweep's lengths, where the plan may trade cluster
    size for co-residency (idle splits included): one cluster per group."""
    s, cs = da.splits_for(1, 16, 16, 128, kv_len, kv_len, torch.float16)
    assert s == cs >= 2
    check_step(ora, W.mha_sweep(kv_len, seed=kv_len % 97), fused, hint=kv_len, what=f"MHA kv {kv_len}")


@pytest.mark.parametrize("kv_len", W.MHA_SWEEP_KV_LENS)
def test_mha_sweep_nan_tail(ora, kv_len):
    check_step(ora, W.mha_sweep(kv_len, seed=2, extra_capacity=64), False, what=f"MHA kv {kv_len} + tail")


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_long_context(ora, fused):
    check_step(ora, W.long_context(seed=3), fused, what="long context 32768")


@pytest.mark.parametrize("seed", [4, 5])
@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_batched_streaming(ora, fused, seed):
    step = W.batched_streaming(seed=seed)
    assert int(step.position_ids.min()) == 0
    check_step(ora, step, fused, what="batched streaming")


@pytest.mark.parametrize("path", ["append+attend", "fused_step", "layers_call"])
def test_s2pro_generation(ora, path):
    """36 layers x 400 steps of append + attend (two calls per layer, one fused
    call per layer, or one decode_step_layers_fwd launch for all 36 layers of
    a step); final caches bit-exact; all 14,400 layer-steps checked against
    the oracle. The oracle of step i reads the final cache: its rows below
    kv_len were already final at step i."""
    g = W.s2pro_generation(seed=6)
    dev = "cuda"
    shape = (g.layers, g.B, g.n_kv_head, g.capacity, g.head_dim)
    kc = W.nan_like(shape, g.dtype, device=dev)
    vc = W.nan_like(shape, g.dtype, device=dev)
    kc[:, :, :, :g.prompt] = g.k_prefix.to(dev)
    vc[:, :, :, :g.prompt] = g.v_prefix.to(dev)
    q, kn, vn = g.q.to(dev), g.k_new.to(dev), g.v_new.to(dev)
    outs = torch.empty((g.steps, g.layers, g.B, g.n_head, g.head_dim), dtype=q.dtype, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = da.alloc_workspace(g.layers * g.B, g.n_head, g.n_kv_head, g.head_dim, g.capacity)
    for i in range(g.steps):
        pos = torch.full((g.B,), g.position(i), dtype=torch.int32, device=dev)
        kv = pos + 1
        if path == "layers_call":
            da.decode_step_layers_fwd(q[i], kc, vc, kn[i], vn[i], pos, out=outs[i], workspace=ws,
                                      max_kv_len_hint=g.position(i) + 1, err_flag=err)
            continue
        for layer in range(g.layers):
            if path == "fused_step":
                da.decode_step_fwd(q[i, layer], kc[layer], vc[layer], kn[i, layer], vn[i, layer], pos,
                                   out=outs[i, layer], workspace=ws, max_kv_len_hint=g.position(i) + 1,
                                   err_flag=err)
            else:
                da.kvcache_append(kc[layer], vc[layer], kn[i, layer], vn[i, layer], pos, err_flag=err)
                da.decode_attn_fwd(q[i, layer], kc[layer], vc[layer], kv, out=outs[i, layer], workspace=ws,
                                   max_kv_len_hint=g.position(i) + 1, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    end = g.prompt + g.steps
    k_full = torch.cat([g.k_prefix, g.k_new.permute(1, 2, 3, 0, 4)], dim=3)  # [layers, B, Hkv, end, D]
    v_full = torch.cat([g.v_prefix, g.v_new.permute(1, 2, 3, 0, 4)], dim=3)
    assert np.array_equal(bits(kc[:, :, :, :end]), bits(k_full)), "K cache prefix"
    assert np.array_equal(bits(vc[:, :, :, :end]), bits(v_full)), "V cache prefix"
    assert bool(torch.isnan(kc[:, :, :, end:].float()).all()) and bool(torch.isnan(vc[:, :, :, end:].float()).all())
    got = outs.cpu()
    q_bits = bits(g.q)
    worst = {"rel_frob": 0.0, "max_abs": 0.0}
    for layer in range(g.layers):
        kb, vb = bits(k_full[layer]), bits(v_full[layer])
        for i in range(g.steps):
            L = g.position(i) + 1
            ref = ora.decode_attn(q_bits[i, layer], kb, vb, np.array([L], np.int32), g.n_head, g.n_kv_head,
                                  g.dtype, threads=THREADS)
            r = assert_close(got[i, layer], ref, f"step {i} layer {layer}")
            worst = {k: max(worst[k], r[k]) for k in worst}
    assert worst["rel_frob"] <= 5e-3


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,H,Hkv", [(64, 4, 1), (128, 16, 16), (128, 32, 8), (64, 16, 8), (128, 8, 1), (64, 8, 8)])
def test_position_zero_returns_v0_bit_exact(dtype, D, H, Hkv):
    """kv_len 1 -> softmax over one entry -> out = V[0], bit for bit."""
    step = W.decode_step(3, H, Hkv, D, 300, dtype, [0, 0, 0], seed=7)
    for fused in FUSED:
        d, out, err = gpu_step(step, fused)
        assert err == 0
        G = H // Hkv
        v0 = d.v_cache[:, :, 0, :].repeat_interleave(G, dim=1)
        assert torch.equal(out.view(torch.int16), v0.contiguous().view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_edge_lengths(ora, dtype, D, G):
    """Lengths at and around tile and split boundaries, ragged across the
    batch, with a NaN tail; both call styles."""
    tile = 8192 // (2 * D)
    Hkv = 2
    # 8-row steps (the tensor-core instances copy partial K tiles in 8-row
    # boxes) and the 64- and 128-row tile edges
    lens = [1, 2, 7, 8, 9, tile - 1, tile, tile + 1, 63, 64, 65, 127, 129, 2 * tile + 3, 1000, 1531]
    cap = max(lens) + 7
    pos = [L - 1 for L in lens]
    step = W.decode_step(len(lens), G * Hkv, Hkv, D, cap, dtype, pos, seed=D * 10 + G)
    for fused in FUSED:
        check_step(ora, step, fused, what=f"{dtype} D{D} G{G} fused={fused}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_many_groups_four_heads_per_kv_head(ora, dtype, D):
    """More (sequence, KV head) groups than SMs with four query heads per KV
    head: one CTA per group, run by the two-CTAs-per-SM kernel; ragged
    lengths with 8-row and tile edges, NaN tail, both call styles."""
    B, Hkv = 40, 4
    rng = np.random.default_rng(D + (1 if dtype == "bf16" else 0))
    lens = [1, 7, 8, 9, 63, 64, 65, 127, 128, 129, 700] + rng.integers(1, 701, B - 11).tolist()
    step = W.decode_step(B, 4 * Hkv, Hkv, D, 707, dtype, [L - 1 for L in lens], seed=90 + D)
    for fused in FUSED:
        check_step(ora, step, fused, what=f"{dtype} D{D} B{B} fused={fused}")


# (B, n_head, n_kv_head, head_dim, capacity, kernel): one case per kernel and
# group size, lengths ragged up to the capacity, bound = capacity.
KERNEL_CASES = [
    (1, 32, 8, 128, 2048, "cuda_cores"),          # 3 tiles per CTA
    (1, 32, 8, 128, 20000, "tensor_cores"),       # 17 tiles per CTA
    (1, 32, 8, 64, 40000, "tensor_cores"),
    (1, 16, 2, 128, 70000, "tensor_cores"),       # eight heads per KV head
    (1, 16, 2, 64, 140000, "tensor_cores"),
    (40, 16, 4, 128, 700, "tensor_cores_paired"),  # 160 groups, one CTA each
    (40, 16, 4, 64, 700, "tensor_cores_paired"),
    (24, 64, 8, 128, 700, "tensor_cores"),        # 192 groups of eight heads: no paired kernel
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", KERNEL_CASES, ids=[f"{c[5]}-G{c[1] // c[2]}-D{c[3]}-B{c[0]}" for c in KERNEL_CASES])
def test_each_kernel(ora, dtype, case):
    """Every decode kernel the library chooses between, against the oracle:
    the case must select the kernel it is meant to cover."""
    B, H, Hkv, D, cap, kernel = case
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    assert da.kernel_for(B, H, Hkv, D, cap, cap, tdt) == kernel
    rng = np.random.default_rng(cap + D + B)
    lens = [cap] + rng.integers(1, cap + 1, B - 1).tolist()
    step = W.decode_step(B, H, Hkv, D, cap, dtype, [L - 1 for L in lens], seed=cap % 1000 + D)
    for fused in FUSED:
        check_step(ora, step, fused, hint=cap, what=f"{kernel} {dtype} G{H // Hkv} D{D} fused={fused}")


def test_capacity_one_and_full(ora):
    check_step(ora, W.decode_step(2, 8, 2, 128, 1, "bf16", [0, 0], seed=8), True, what="capacity 1")
    check_step(ora, W.decode_step(2, 8, 2, 64, 777, "f16", [776, 776], seed=9), False, what="full capacity")


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("kv_len", W.MHA_SWEEP_KV_LENS)
def test_mha_sweep_exact_bound(ora, kv_len, fused):
    """The length bound given as the exact length, as the benchmark calls it:
    one sequence, so the first tiles are issued before the length is read."""
    check_step(ora, W.mha_sweep(kv_len, seed=11), fused, hint=kv_len, what=f"MHA kv {kv_len} exact bound")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,H,Hkv", [(128, 16, 16), (128, 32, 8), (64, 8, 1)])
def test_single_sequence_bounds(ora, dtype, D, H, Hkv):
    """One sequence with a bound equal to, above and below its length: tiles
    issued from the bound are kept only when it is exact, and discarded
    otherwise (the NaN tail would show any discarded row that got used)."""
    cap = 5000
    for L in (1, 2, 63, 64, 65, 300, 1531, 4999):
        step = W.decode_step(1, H, Hkv, D, cap, dtype, [L - 1], seed=L + D)
        for hint in sorted({L, L + 1, L + 100, max(1, L - 1), cap}):
            for fused in FUSED:
                check_step(ora, step, fused, hint=hint, what=f"{dtype} D{D} H{H}/{Hkv} L{L} bound {hint} fused={fused}")


@pytest.mark.parametrize("hint", [1, 64, 5000, 100000])
def test_hint_only_sizes_the_launch(ora, hint):
    """Any max_kv_len_hint gives the same correct result, even one below the
    real lengths."""
    step = W.decode_step(2, 32, 8, 128, 4096, "bf16", [4095, 1200], seed=10)
    check_step(ora, step, False, hint=hint, what=f"hint {hint}")
    check_step(ora, step, True, hint=hint, what=f"fused hint {hint}")


def test_fused_step_matches_two_calls_bitwise():
    step = W.batched_streaming(seed=11)
    d1, o1, e1 = gpu_step(step, False)
    d2, o2, e2 = gpu_step(step, True)
    assert e1 == e2 == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(d1.k_cache.view(torch.int16), d2.k_cache.view(torch.int16))
    assert torch.equal(d1.v_cache.view(torch.int16), d2.v_cache.view(torch.int16))


def test_deterministic():
    step = W.long_context(seed=12, kv_len=20000)
    outs = [gpu_step(step, False)[1] for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_empty_batch():
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.empty(0, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.empty(0, dtype=torch.int32, device="cuda")
    out = da.decode_attn_fwd(q, kc, kc.clone(), kv)
    assert out.shape == (0, 8, 128)


def test_invalid_lengths_give_nan_rows_and_error_bits(ora):
    step = W.decode_step(3, 8, 2, 128, 100, "f16", [50, 5, 50], seed=13)
    d = step.to("cuda")
    kv_len = torch.tensor([0, 6, 101], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, kv_len, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == da.DA_DEVERR_KV_LEN
    assert bool(torch.isnan(out[0].float()).all()) and bool(torch.isnan(out[2].float()).all())
    # kv_len 6 of sequence 1 includes its NaN row 5 (the unwritten append
    # slot): a NaN inside the prefix propagates on both sides
    ref = ora.decode_attn(bits(step.q[1:2]), bits(step.k_cache[1:2]), bits(step.v_cache[1:2]),
                          np.array([6], np.int32), 8, 2, "f16")
    assert np.all(np.isnan(ref)) and bool(torch.isnan(out[1].float()).all())
    kv_len = torch.tensor([0, 5, 101], dtype=torch.int32, device="cuda")
    err.zero_()
    out = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, kv_len, err_flag=err)
    ref = ora.decode_attn(bits(step.q[1:2]), bits(step.k_cache[1:2]), bits(step.v_cache[1:2]),
                          np.array([5], np.int32), 8, 2, "f16")
    assert_close(out[1:2], ref, "valid row among invalid ones")
    assert int(err.item()) == da.DA_DEVERR_KV_LEN


def test_invalid_positions_skip_the_write(ora):
    step = W.decode_step(3, 8, 2, 64, 40, "bf16", [10, 3, 10], seed=14)
    for fused in FUSED:
        d = step.to("cuda")
        before_k = d.k_cache.clone()
        pos = torch.tensor([-1, 3, 40], dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, pos, err_flag=err)
        else:
            da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, pos, err_flag=err)
            out = None
        torch.cuda.synchronize()
        expect = da.DA_DEVERR_POSITION | (da.DA_DEVERR_KV_LEN if fused else 0)
        assert int(err.item()) == expect
        assert torch.equal(d.k_cache[0].view(torch.int16), before_k[0].view(torch.int16))
        assert torch.equal(d.k_cache[2].view(torch.int16), before_k[2].view(torch.int16))
        assert torch.equal(d.k_cache[1, :, 3].view(torch.int16), d.k_new[1].view(torch.int16))
        if fused:
            assert bool(torch.isnan(out[0].float()).all()) and bool(torch.isnan(out[2].float()).all())
            assert bool(torch.isfinite(out[1].float()).all())


def test_no_writes_outside_out_and_workspace():
    step = W.long_context(seed=15, kv_len=9000, capacity=9000)
    d = step.to("cuda")
    B, H, D = d.q.shape
    guard = 64
    out_buf = torch.full((B * H * D + 2 * guard,), 12345, dtype=torch.int16, device="cuda")
    out = out_buf[guard:guard + B * H * D].view(torch.bfloat16).view(B, H, D)
    n = da.decode_attn_workspace_size(B, H, 8, D, d.capacity)
    assert n > 0
    ws_buf = torch.full((n + 2 * 256,), 7, dtype=torch.uint8, device="cuda")
    ws = ws_buf[256:256 + n]
    da.workspace_init(ws)
    da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), out=out, workspace=ws)
    torch.cuda.synchronize()
    assert bool((out_buf[:guard] == 12345).all()) and bool((out_buf[-guard:] == 12345).all())
    assert bool((ws_buf[:256] == 7).all()) and bool((ws_buf[-256:] == 7).all())


def test_side_stream(ora):
    step = W.decode_step(2, 16, 8, 128, 3000, "bf16", [2999, 17], seed=16)
    kb, vb, ref = oracle_step(ora, step)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = step.to("cuda")
        out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    s.synchronize()
    assert_close(out, ref, "side stream")


def test_small_workspace_is_rejected():
    step = W.long_context(seed=17, kv_len=20000, capacity=20000).to("cuda")
    assert da.decode_attn_workspace_size(1, 32, 8, 128, 20000) > 16
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_fwd(step.q, step.k_cache, step.v_cache, step.kv_len.contiguous(),
                           workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -4


def test_layers_call_is_one_batched_launch(ora):
    """decode_step_layers_fwd over stacked layers gives, bit for bit, the
    caches and outputs of one decode_step_fwd on the flattened
    [layers * B, ...] batch (positions repeated per layer), and every layer
    matches the oracle."""
    layers, B, H, Hkv, D, cap, dt = 6, 2, 32, 8, 128, 1000, "bf16"
    pos = [999, 400]
    steps = [W.decode_step(B, H, Hkv, D, cap, dt, pos, seed=60 + l) for l in range(layers)]
    stack = lambda name: torch.stack([getattr(s, name) for s in steps]).cuda()  # noqa: E731
    q, kc, vc, kn, vn = (stack(n) for n in ("q", "k_cache", "v_cache", "k_new", "v_new"))
    p = steps[0].position_ids.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc2, vc2 = kc.clone(), vc.clone()
    out = da.decode_step_layers_fwd(q, kc, vc, kn, vn, p, max_kv_len_hint=cap, err_flag=err)
    flat = lambda t: t.reshape(layers * B, *t.shape[2:])  # noqa: E731
    ref = da.decode_step_fwd(flat(q), flat(kc2), flat(vc2), flat(kn), flat(vn), p.repeat(layers),
                             max_kv_len_hint=cap).view(q.shape)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
    for l in range(layers):
        kb, vb, o = oracle_step(ora, steps[l])
        assert np.array_equal(bits(kc[l]), kb) and np.array_equal(bits(vc[l]), vb)
        assert_close(out[l], o, f"layer {l}")


def test_layers_call_rejects_before_any_write():
    """An argument error of decode_step_layers_fwd (here a workspace sized for
    one layer's batch, too small for the whole stack) is reported before the
    launch: no layer's cache or output is touched."""
    layers, B, H, Hkv, D, cap = 4, 1, 32, 8, 128, 20000
    steps = [W.decode_step(B, H, Hkv, D, cap, "bf16", [19999], seed=70 + l) for l in range(layers)]
    stack = lambda name: torch.stack([getattr(s, name) for s in steps]).cuda()  # noqa: E731
    q, kc, vc, kn, vn = (stack(n) for n in ("q", "k_cache", "v_cache", "k_new", "v_new"))
    p = steps[0].position_ids.cuda()
    need_one = da.decode_attn_workspace_size(B, H, Hkv, D, cap)
    need_all = da.decode_attn_workspace_size(layers * B, H, Hkv, D, cap)
    small = torch.zeros(max(need_one, 16), dtype=torch.uint8, device="cuda")
    kc0, vc0 = kc.clone(), vc.clone()
    out = torch.full_like(q, 7.0)
    if need_all > small.numel():
        with pytest.raises(da.DecodeAttnError) as e:
            da.decode_step_layers_fwd(q, kc, vc, kn, vn, p, out=out, workspace=small, max_kv_len_hint=cap)
        assert e.value.status == -4
    # a misaligned k_new (all layers share one alignment): rejected before the launch
    lib = da.load_library()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.decode_step_layers_fwd(ptr(q), ptr(kc), ptr(vc), ctypes.c_void_p(kn.data_ptr() + 4), ptr(vn), ptr(p),
                                    layers, B, H, Hkv, D, cap, 0.1, ptr(out), ptr(small), small.numel(), cap, 1,
                                    None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == -6
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), kc0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc0.view(torch.int16))
    assert bool((out.float() == 7.0).all())


def test_binding_checks_flags_and_counts_workspace_bytes(ora):
    """The binding rejects an error flag that is not int32 and passes a
    workspace's size in bytes whatever its element type."""
    step = W.long_context(seed=18, kv_len=9000, capacity=9000)
    kb, vb, ref = oracle_step(ora, step)
    d = step.to("cuda")
    with pytest.raises(ValueError):
        da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids,
                          err_flag=torch.zeros(1, dtype=torch.int64, device="cuda"))
    da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    n = da.decode_attn_workspace_size(1, step.n_head, step.n_kv_head, step.head_dim, step.capacity)
    assert n > 16
    ws = torch.zeros((n + 15) // 16, 4, dtype=torch.float32, device="cuda")
    out = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), workspace=ws,
                             max_kv_len_hint=step.capacity)
    torch.cuda.synchronize()
    assert np.array_equal(bits(d.k_cache), kb) and np.array_equal(bits(d.v_cache), vb)
    assert_close(out, ref, "float32 workspace")


@pytest.mark.parametrize("world", [2, 3])
def test_kv_head_shards_concatenate_to_the_full_step(ora, world):
    """Each rank's block of KV heads (decode_attn_shard_heads) run through the
    fused step on its own contiguous tensors, one after another on this GPU:
    the outputs side by side on the head axis, and the cache blocks, are the
    full step's (outputs within tolerance: each block has its own split
    plan), and match the oracle."""
    step = W.decode_step(2, 32, 8, 128, 5000, "bf16", [4999, 2500], seed=85)
    kb, vb, ref = oracle_step(ora, step)
    outs, kcs, vcs = [], [], []
    for rank in range(world):
        kv0, nkv, h0, nh = da.shard_heads(step.n_head, step.n_kv_head, world, rank)
        part = W.DecodeStep(step.q[:, h0:h0 + nh].contiguous(), step.k_cache[:, kv0:kv0 + nkv].contiguous(),
                            step.v_cache[:, kv0:kv0 + nkv].contiguous(), step.k_new[:, kv0:kv0 + nkv].contiguous(),
                            step.v_new[:, kv0:kv0 + nkv].contiguous(), step.position_ids, nh, nkv, step.dtype)
        d, out, err = gpu_step(part, True, hint=5000)
        assert err == 0
        outs.append(out.cpu())
        kcs.append(bits(d.k_cache))
        vcs.append(bits(d.v_cache))
    assert np.array_equal(np.concatenate(kcs, axis=1), kb) and np.array_equal(np.concatenate(vcs, axis=1), vb)
    got = torch.cat(outs, dim=1)
    assert_close(got, ref, f"{world} shards vs oracle")
    _, full, _ = gpu_step(step, True, hint=5000)
    assert_close(got, full.double().cpu().numpy(), f"{world} shards vs the full step")
