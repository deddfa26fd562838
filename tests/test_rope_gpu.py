"""GPU parity of the fused step with rotary position embedding
(decode_step_rope_fwd) against the oracle: the oracle rotates q and k_new
(fp32 arithmetic, one rounding to the storage type), appends the rotated key
and v_new, and attends with the rotated q. The cache must match bit for bit,
the output within the method's tolerances."""
import numpy as np
import pytest
import torch

import decode_attention_static_gb300 as da
import workloads as W
from gpu_helpers import THREADS, assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build_library()
    da.load_library()


def tables(step: W.DecodeStep, kind: str, rows: int | None = None):
    rows = rows or step.capacity
    if kind == "ladder":
        return W.rope_tables(rows, step.head_dim)
    return W.random_rope_tables(rows, step.head_dim, seed=rows + step.head_dim)


def oracle_rope_step(ora, step: W.DecodeStep, cos, sin):
    pos = step.position_ids.numpy()
    q_rot, bad_q = ora.rope(bits(step.q), cos.numpy(), sin.numpy(), pos, step.dtype)
    k_rot, bad_k = ora.rope(bits(step.k_new), cos.numpy(), sin.numpy(), pos, step.dtype)
    assert bad_q == 0 and bad_k == 0
    kb, vb = bits(step.k_cache).copy(), bits(step.v_cache).copy()
    ora.kvcache_append(kb, vb, k_rot, bits(step.v_new), pos)
    out = ora.decode_attn(q_rot, kb, vb, step.kv_len.numpy(), step.n_head, step.n_kv_head, step.dtype,
                          threads=THREADS)
    return q_rot, k_rot, kb, vb, out


def gpu_rope_step(step: W.DecodeStep, cos, sin, hint: int = 0):
    d = step.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = da.decode_step_rope_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, cos.cuda(), sin.cuda(),
                                  d.position_ids, max_kv_len_hint=hint, err_flag=err)
    torch.cuda.synchronize()
    return d, out, int(err.item())


def check_rope_step(ora, step, kind="random", hint=0, what=""):
    cos, sin = tables(step, kind)
    _, _, kb, vb, ref = oracle_rope_step(ora, step, cos, sin)
    d, out, err = gpu_rope_step(step, cos, sin, hint)
    assert err == 0, f"{what}: device error flag {err}"
    assert np.array_equal(bits(d.k_cache), kb), f"{what}: K cache differs from the oracle's rotated append"
    assert np.array_equal(bits(d.v_cache), vb), f"{what}: V cache differs from the oracle's append"
    return assert_close(out, ref, what)


def test_tiny_gqa(ora):
    check_rope_step(ora, W.tiny_gqa(seed=0), "ladder", what="tiny GQA")


@pytest.mark.parametrize("kv_len", W.MHA_SWEEP_KV_LENS)
@pytest.mark.parametrize("exact", [False, True], ids=["no bound", "exact bound"])
def test_mha_sweep(ora, kv_len, exact):
    check_rope_step(ora, W.mha_sweep(kv_len, seed=21), "ladder", hint=kv_len if exact else 0,
                    what=f"MHA kv {kv_len}")


def test_long_context(ora):
    check_rope_step(ora, W.long_context(seed=22), "ladder", hint=32768, what="long context")


def test_batched_streaming(ora):
    s = W.batched_streaming(seed=23)
    check_rope_step(ora, s, "random", hint=int(s.position_ids.max()) + 1, what="batched streaming")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,G", [(64, 1), (64, 4), (128, 2), (128, 8)])
def test_bounds_and_lengths(ora, dtype, D, G):
    """One sequence at lengths around tile boundaries, with bounds equal to,
    above and below the length (early tiles kept or discarded, the rotated row
    in an early tile or in a later one), random rotations."""
    Hkv, cap = 2, 1600
    for L in (1, 2, 64, 65, 129, 1531):
        step = W.decode_step(1, G * Hkv, Hkv, D, cap, dtype, [L - 1], seed=L + D + G)
        for hint in sorted({L, L + 1, max(1, L - 1), cap}):
            check_rope_step(ora, step, "random", hint=hint, what=f"{dtype} D{D} G{G} L{L} bound {hint}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_position_zero_returns_v_new(dtype):
    """At position 0 the ladder tables hold cos = 1, sin = 0: the rotation is
    the identity, the only visible row is the appended one, so out = v_new."""
    step = W.decode_step(3, 16, 4, 128, 64, dtype, [0, 0, 0], seed=31)
    cos, sin = W.rope_tables(64, 128)
    d, out, err = gpu_rope_step(step, cos, sin, hint=1)
    assert err == 0
    want = d.v_new.repeat_interleave(4, dim=1)
    assert torch.equal(out.view(torch.int16), want.contiguous().view(torch.int16))


@pytest.mark.parametrize("shape", [(2, 1500, [1499, 700], 128, "cuda_cores"), (1, 20000, [19999], 128, "tensor_cores"),
                                   (1, 40000, [39998], 64, "tensor_cores"), (40, 700, None, 128, "tensor_cores_paired")],
                         ids=lambda s: f"{s[4]}-D{s[3]}")
def test_matches_unrotated_step_on_rotated_inputs(ora, shape):
    """The fused rotation is bit-identical to rotating q and k_new with the
    oracle and running the plain fused step: same cache, same output bits
    (32 / 8 heads, bf16; each of the kernels the library chooses between)."""
    B, cap, pos, D, kernel = shape
    if pos is None:
        pos = np.random.default_rng(5).integers(0, cap, B).tolist()
    assert da.kernel_for(B, 32, 8, D, cap, 0, torch.bfloat16, rotary=True) == kernel
    assert da.kernel_for(B, 32, 8, D, cap, 0, torch.bfloat16) == kernel
    step = W.decode_step(B, 32, 8, D, cap, "bf16", pos, seed=32)
    cos, sin = tables(step, "random")
    q_rot, k_rot, _, _, _ = oracle_rope_step(ora, step, cos, sin)
    d_rope, out_rope, err = gpu_rope_step(step, cos, sin)
    assert err == 0
    plain = W.DecodeStep(torch.from_numpy(q_rot.view(np.int16)).view(step.q.dtype), step.k_cache.clone(),
                         step.v_cache.clone(), torch.from_numpy(k_rot.view(np.int16)).view(step.k_new.dtype),
                         step.v_new, step.position_ids, step.n_head, step.n_kv_head, step.dtype)
    d = plain.to("cuda")
    out_plain = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids)
    torch.cuda.synchronize()
    assert torch.equal(d_rope.k_cache.view(torch.int16), d.k_cache.view(torch.int16))
    assert torch.equal(out_rope.view(torch.int16), out_plain.view(torch.int16))


def test_rejects_short_or_missing_tables():
    step = W.decode_step(1, 8, 2, 64, 100, "f16", [10], seed=33).to("cuda")
    cos, sin = W.rope_tables(99, 64)
    with pytest.raises(da.DecodeAttnError):
        da.decode_step_rope_fwd(step.q, step.k_cache, step.v_cache, step.k_new, step.v_new, cos.cuda(), sin.cuda(),
                                step.position_ids)
