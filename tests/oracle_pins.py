"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics that
the oracle must reproduce, each checked against something other than the
oracle itself (a closed form, a library routine, brute force in plain Python,
an invariant of the definition, or bit-level equality with the inputs).

Every pin is a function of an ``oracle.Oracle`` so that the same suite can
run against deliberately broken builds of the oracle source (see
test_oracle_mutants.py). Run as a script, it executes every pin against the
library given on the command line and prints a JSON map pin -> "ok"/error.
"""
from __future__ import annotations

import json
import math
import sys

import numpy as np
import torch
import torch.nn.functional as F

import workloads as W

F16_NAN = 0x7E00
BF16_NAN = 0x7FC0


def _exact_f64(t: torch.Tensor) -> np.ndarray:
    """Decode 16-bit values with torch's own conversion (exact in fp64)."""
    return t.detach().to(torch.float64).numpy()


def _case(B, H, Hkv, D, cap, dtype, kv_len, seed, finite_tail=False):
    """Random q/K/V; rows >= kv_len[b] NaN unless finite_tail."""
    gen = W.generator(seed)
    q = W.randn((B, H, D), dtype, gen)
    k = W.randn((B, Hkv, cap, D), dtype, gen)
    v = W.randn((B, Hkv, cap, D), dtype, gen)
    kv_len = np.asarray(kv_len, dtype=np.int32)
    k_nan, v_nan = k.clone(), v.clone()
    for b in range(B):
        L = int(kv_len[b])
        if L < cap:
            k_nan[b, :, L:] = W.nan_like((Hkv, cap - L, D), dtype)
            v_nan[b, :, L:] = W.nan_like((Hkv, cap - L, D), dtype)
    if finite_tail:
        return q, k, v, kv_len
    return q, k_nan, v_nan, kv_len


def _sdpa_prefix(q, k, v, kv_len, scale):
    """torch SDPA in float64 on the sliced prefix with enable_gqa=True: the
    call of the patched forward_step in VoxCPM issue #395, section 4.1."""
    B, H, D = q.shape
    out = np.empty((B, H, D))
    for b in range(B):
        L = int(kv_len[b])
        qb = q[b:b + 1].to(torch.float64).unsqueeze(2)  # [1, H, 1, D]
        kb = k[b:b + 1, :, :L].to(torch.float64)
        vb = v[b:b + 1, :, :L].to(torch.float64)
        o = F.scaled_dot_product_attention(qb, kb, vb, scale=scale, enable_gqa=True)
        out[b] = o[0, :, 0].numpy()
    return out


def _sdpa_masked_full(q, k, v, kv_len, scale):
    """torch SDPA in float64 over the full capacity with the boolean mask
    arange(capacity) <= position_id: the original forward_step of VoxCPM
    issue #395, section 2.1."""
    B, H, D = q.shape
    cap = k.shape[2]
    out = np.empty((B, H, D))
    for b in range(B):
        pos = int(kv_len[b]) - 1
        mask = (torch.arange(cap) <= pos).view(1, 1, 1, cap)
        qb = q[b:b + 1].to(torch.float64).unsqueeze(2)
        o = F.scaled_dot_product_attention(qb, k[b:b + 1].to(torch.float64), v[b:b + 1].to(torch.float64),
                                           attn_mask=mask, scale=scale, enable_gqa=True)
        out[b] = o[0, :, 0].numpy()
    return out


def _assert_close(a, b, rtol, atol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        raise AssertionError(f"{what}: shape {a.shape} vs {b.shape}")
    if not np.all(np.isfinite(a)):
        raise AssertionError(f"{what}: non-finite values in oracle output")
    err = np.abs(a - b)
    tol = atol + rtol * np.abs(b)
    if not np.all(err <= tol):
        i = int(np.argmax(err - tol))
        raise AssertionError(f"{what}: max err {err.max():.3e} at flat {i} ({a.flat[i]!r} vs {b.flat[i]!r})")


def _bits(t):
    return W.raw_bits(t)


# ---------------------------------------------------------------------------
# Pins.

def pin_decoders_exhaustive(ora):
    """All 65536 fp16 and bf16 bit patterns decode as numpy/torch decode them."""
    allbits = np.arange(65536, dtype=np.uint16)
    ref16 = allbits.view(np.float16).astype(np.float64)
    got16 = ora.decode_bits(allbits, "f16")
    refbf = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    gotbf = ora.decode_bits(allbits, "bf16")
    for name, ref, got in (("f16", ref16, got16), ("bf16", refbf, gotbf)):
        nan_r, nan_g = np.isnan(ref), np.isnan(got)
        if not np.array_equal(nan_r, nan_g):
            raise AssertionError(f"{name}: NaN patterns differ")
        if not np.array_equal(ref[~nan_r], got[~nan_g]):
            bad = np.nonzero(ref[~nan_r] != got[~nan_g])[0][:4]
            raise AssertionError(f"{name}: values differ at {bad}")
        # signed zeros must keep their sign
        if not np.array_equal(np.signbit(ref[~nan_r]), np.signbit(got[~nan_g])):
            raise AssertionError(f"{name}: sign bits differ")


def pin_position0_returns_v0(ora):
    """position_id 0 -> the slice [:1] -> softmax over one entry is the
    identity, so out = V[0] exactly (VoxCPM issue #395, section 3)."""
    for dtype in ("f16", "bf16"):
        B, H, Hkv, D, cap = 3, 8, 2, 64, 16
        q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [1, 1, 1], seed=11)
        out = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype)
        v0 = _exact_f64(v[:, :, 0, :])  # [B, Hkv, D]
        G = H // Hkv
        for h in range(H):
            if not np.array_equal(out[:, h], v0[:, h // G]):
                raise AssertionError(f"{dtype}: head {h} is not V[0] of KV head {h // G}")


def pin_prefix_equals_masked_full_capacity(ora):
    """Attention on the active prefix equals attention over the whole
    capacity with the tail masked (fish-speech issue #1310, section 1;
    VoxCPM issue #395, sections 2.1 and 3). The oracle sees a NaN tail, the
    library routine a finite one."""
    for dtype, (B, H, Hkv, D, cap, kv) in (("f16", (2, 4, 1, 64, 40, [37, 5])),
                                           ("bf16", (3, 8, 2, 32, 24, [24, 1, 13]))):
        q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, kv, seed=5, finite_tail=True)
        _, k_nan, v_nan, _ = _case(B, H, Hkv, D, cap, dtype, kv, seed=5)
        scale = 1.0 / math.sqrt(D)
        got = ora.decode_attn(_bits(q), _bits(k_nan), _bits(v_nan), kv_len, H, Hkv, dtype, scale)
        ref = _sdpa_masked_full(q, k, v, kv_len, scale)
        _assert_close(got, ref, 1e-12, 1e-13, f"{dtype} masked full capacity")


def pin_sdpa_prefix_slice(ora):
    """Random GQA and MHA shapes against torch SDPA (float64, enable_gqa) on
    the sliced prefix, the patched call of VoxCPM issue #395, section 4.1."""
    shapes = [("f16", 1, 4, 1, 64, 256, [37]), ("f16", 1, 16, 16, 128, 64, [64]),
              ("bf16", 2, 32, 8, 128, 48, [48, 17]), ("bf16", 4, 16, 8, 128, 33, [1, 33, 2, 20]),
              ("f16", 2, 6, 3, 16, 9, [9, 4])]
    for i, (dtype, B, H, Hkv, D, cap, kv) in enumerate(shapes):
        q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, kv, seed=100 + i)
        scale = 1.0 / math.sqrt(D)
        got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale)
        ref = _sdpa_prefix(q, k, v, kv_len, scale)
        _assert_close(got, ref, 1e-12, 1e-13, f"shape {i}")


def pin_gqa_equals_expanded_mha(ora):
    """Grouped KV heads give exactly what repeat_interleave-expanded MHA
    gives (fish-speech issue #1310, section 2, steps 4-5)."""
    for dtype in ("f16", "bf16"):
        B, H, Hkv, D, cap = 2, 12, 3, 32, 20
        q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [20, 7], seed=3)
        G = H // Hkv
        got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype)
        ke, ve = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
        ref = ora.decode_attn(_bits(q), _bits(ke), _bits(ve), kv_len, H, H, dtype)
        if not np.array_equal(got, ref):
            raise AssertionError(f"{dtype}: GQA differs from expanded MHA")


def pin_equal_scores_give_mean(ora):
    """Equal scores (q = 0, or scale = 0, or identical key rows) make the
    softmax uniform, so out is the plain mean of V over the prefix."""
    B, H, Hkv, D, cap, dtype = 2, 4, 2, 16, 12, "bf16"
    q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [12, 5], seed=21)
    G = H // Hkv
    vmean = np.stack([_exact_f64(v[b, :, :kv_len[b]]).mean(axis=1) for b in range(B)])  # [B, Hkv, D]
    ref = np.repeat(vmean, G, axis=1)
    zeros = torch.zeros_like(q)
    got = ora.decode_attn(_bits(zeros), _bits(k), _bits(v), kv_len, H, Hkv, dtype)
    _assert_close(got, ref, 1e-13, 1e-15, "q = 0")
    got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale=0.0)
    _assert_close(got, ref, 1e-13, 1e-15, "scale = 0")
    k_same = k.clone()
    k_same[:, :, :, :] = k[:, :, :1, :]
    got = ora.decode_attn(_bits(q), _bits(k_same), _bits(v), kv_len, H, Hkv, dtype)
    _assert_close(got, ref, 1e-13, 1e-15, "identical keys")


def pin_two_keys_logistic(ora):
    """With two visible rows the softmax weights are the logistic function
    of the score difference: out = V0 / (1 + e^(x1 - x0)) + V1 / (1 + e^(x0 - x1))."""
    B, H, Hkv, D, cap, dtype = 1, 2, 1, 8, 6, "f16"
    q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [2], seed=8)
    scale = 0.37
    got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale)
    qd, kd, vd = _exact_f64(q), _exact_f64(k), _exact_f64(v)
    for h in range(H):
        x0 = scale * math.fsum(qd[0, h] * kd[0, 0, 0])
        x1 = scale * math.fsum(qd[0, h] * kd[0, 0, 1])
        w0 = 1.0 / (1.0 + math.exp(x1 - x0))
        w1 = 1.0 / (1.0 + math.exp(x0 - x1))
        _assert_close(got[0, h], w0 * vd[0, 0, 0] + w1 * vd[0, 0, 1], 1e-13, 1e-15, f"head {h}")


def pin_dominant_key_selects_its_value(ora):
    """A key whose score exceeds every other by thousands takes all the
    weight: out = V[j*] (the softmax limit)."""
    B, H, Hkv, D, cap, dtype = 1, 1, 1, 32, 10, "bf16"
    q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [10], seed=9)
    for jstar in (0, 6, 9):  # first, middle and last visible row
        q = k[:, :, jstar, :].clone()  # q = K[j*]: the largest self-similarity
        got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale=200.0)
        if not np.array_equal(got[0, 0], _exact_f64(v[0, 0, jstar])):
            raise AssertionError(f"dominant key {jstar} did not select its value row")


def pin_large_scores_stay_finite(ora):
    """Scores near 1e4 overflow exp() unless the max is subtracted first
    (Cuda-Compute-OSS issue #343, 'Correctness risks': standard
    max-subtracted softmax). Checked against torch SDPA in float64."""
    B, H, Hkv, D, cap, dtype = 2, 4, 2, 64, 30, "f16"
    q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [30, 11], seed=13)
    scale = 50.0
    got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale)
    ref = _sdpa_prefix(q, k, v, kv_len, scale)
    _assert_close(got, ref, 1e-11, 1e-12, "large scores")


def pin_convex_hull_and_permutation(ora):
    """out is a convex combination of the visible V rows (per component within
    [min_j V, max_j V]); permuting the (K_j, V_j) pairs leaves it unchanged."""
    B, H, Hkv, D, cap, dtype = 2, 8, 4, 32, 40, "bf16"
    q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, [40, 23], seed=17)
    got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype)
    G = H // Hkv
    vd = _exact_f64(v)
    for b in range(B):
        L = int(kv_len[b])
        for h in range(H):
            lo = vd[b, h // G, :L].min(axis=0)
            hi = vd[b, h // G, :L].max(axis=0)
            if np.any(got[b, h] < lo - 1e-12) or np.any(got[b, h] > hi + 1e-12):
                raise AssertionError("output outside the convex hull of V")
    perm_k, perm_v = k.clone(), v.clone()
    gen = torch.Generator().manual_seed(1)
    for b in range(B):
        L = int(kv_len[b])
        p = torch.randperm(L, generator=gen)
        perm_k[b, :, :L] = k[b, :, p]
        perm_v[b, :, :L] = v[b, :, p]
    got2 = ora.decode_attn(_bits(q), _bits(perm_k), _bits(perm_v), kv_len, H, Hkv, dtype)
    _assert_close(got2, got, 1e-12, 1e-14, "permuted prefix")


def pin_brute_force_python(ora):
    """Tiny shapes against a plain-Python evaluation of the definition with
    math.fsum and math.exp (inputs decoded by torch)."""
    for seed, (dtype, B, H, Hkv, D, cap, kv) in enumerate([("f16", 2, 2, 1, 4, 5, [5, 3]),
                                                           ("bf16", 1, 4, 2, 8, 5, [4]),
                                                           ("f16", 2, 3, 3, 2, 3, [1, 2])]):
        q, k, v, kv_len = _case(B, H, Hkv, D, cap, dtype, kv, seed=40 + seed)
        scale = 1.0 / math.sqrt(D)
        got = ora.decode_attn(_bits(q), _bits(k), _bits(v), kv_len, H, Hkv, dtype, scale)
        qd, kd, vd = _exact_f64(q).tolist(), _exact_f64(k).tolist(), _exact_f64(v).tolist()
        G = H // Hkv
        for b in range(B):
            L = int(kv_len[b])
            for h in range(H):
                g = h // G
                xs = [scale * math.fsum(qd[b][h][d] * kd[b][g][j][d] for d in range(D)) for j in range(L)]
                mx = max(xs)
                ws = [math.exp(x - mx) for x in xs]
                z = math.fsum(ws)
                ref = [math.fsum(ws[j] * vd[b][g][j][d] for j in range(L)) / z for d in range(D)]
                _assert_close(got[b, h], ref, 1e-13, 1e-15, f"seed {seed} b {b} h {h}")


def pin_new_row_is_attended(ora):
    """Append at position_id then attend over [0, position_id]: the row just
    written is visible and the row after it is not (VoxCPM issue #395,
    section 4.1; at position_id 1500 the patched path attends 1501 rows,
    section 6.4)."""
    B, H, Hkv, D, cap, dtype = 1, 4, 2, 16, 1504, "bf16"
    step = W.decode_step(B, H, Hkv, D, cap, dtype, [1500], seed=31)
    kc, vc = _bits(step.k_cache).copy(), _bits(step.v_cache).copy()
    bad = ora.kvcache_append(kc, vc, _bits(step.k_new), _bits(step.v_new), step.position_ids.numpy())
    if bad:
        raise AssertionError("in-range position reported as bad")
    kv_len = step.kv_len.numpy()
    if int(kv_len[0]) != 1501:
        raise AssertionError("kv_len must be position_id + 1")
    got = ora.decode_attn(_bits(step.q), kc, vc, kv_len, H, Hkv, dtype)
    if not np.all(np.isfinite(got)):
        raise AssertionError("NaN row 1501 leaked or the new row was not written")
    k_full = step.k_cache.clone()
    v_full = step.v_cache.clone()
    k_full[:, :, 1500] = step.k_new
    v_full[:, :, 1500] = step.v_new
    ref = _sdpa_prefix(step.q, k_full, v_full, kv_len, 1.0 / math.sqrt(D))
    _assert_close(got, ref, 1e-12, 1e-13, "after append")


def pin_append_is_bit_exact(ora):
    """The append copies raw bits into row position_id and touches nothing
    else; NaN payloads elsewhere survive; a position outside [0, capacity) is
    skipped and counted."""
    for dtype, nan_payload in (("f16", 0x7E01), ("bf16", 0x7FC1)):
        B, Hkv, D, cap = 4, 3, 16, 10
        gen = W.generator(2)
        kc = W.randn((B, Hkv, cap, D), dtype, gen)
        vc = W.randn((B, Hkv, cap, D), dtype, gen)
        kb, vb = _bits(kc).copy(), _bits(vc).copy()
        kb[:, :, 7:] = nan_payload
        vb[:, :, 7:] = nan_payload
        k_new = _bits(W.randn((B, Hkv, D), dtype, gen))
        v_new = _bits(W.randn((B, Hkv, D), dtype, gen))
        pos = np.array([0, 9, -1, 10], dtype=np.int32)
        k_after, v_after = kb.copy(), vb.copy()
        bad = ora.kvcache_append(k_after, v_after, k_new, v_new, pos)
        if bad != 2:
            raise AssertionError(f"expected 2 out-of-range positions, got {bad}")
        exp_k, exp_v = kb.copy(), vb.copy()
        for b, p in enumerate(pos):
            if 0 <= p < cap:
                exp_k[b, :, p] = k_new[b]
                exp_v[b, :, p] = v_new[b]
        if not (np.array_equal(k_after, exp_k) and np.array_equal(v_after, exp_v)):
            raise AssertionError(f"{dtype}: cache bits differ from the expected append")


def pin_invalid_kv_len_gives_nan_rows(ora):
    """kv_len outside [1, capacity] is a precondition violation: that
    sequence's rows are NaN and the other sequences are unaffected."""
    B, H, Hkv, D, cap, dtype = 3, 2, 1, 8, 6, "f16"
    q, k, v, _ = _case(B, H, Hkv, D, cap, dtype, [6, 6, 6], seed=4, finite_tail=True)
    # The over-long length sits on the first sequence, so that an oracle
    # that failed to reject it would read the next sequence's finite rows
    # (defined memory) and give finite values instead of NaN.
    got = ora.decode_attn(_bits(q), _bits(k), _bits(v), np.array([7, 4, 0], np.int32), H, Hkv, dtype)
    if not (np.all(np.isnan(got[0])) and np.all(np.isnan(got[2]))):
        raise AssertionError("invalid kv_len rows must be NaN")
    ref = _sdpa_prefix(q[1:2], k[1:2], v[1:2], np.array([4]), 1.0 / math.sqrt(D))
    _assert_close(got[1:2], ref, 1e-12, 1e-13, "valid row")


def pin_encoders_round_to_nearest_even(ora):
    """fp32 -> fp16 / bf16 storage: every finite 16-bit value round-trips bit
    for bit, random fp32 values round as numpy's float16 and torch's bfloat16
    casts do (both round to nearest even), and the midpoint between two
    neighbouring fp16 values goes to the one with an even last bit."""
    allbits = np.arange(65536, dtype=np.uint16)
    for name in ("f16", "bf16"):
        vals = ora.decode_bits(allbits, name)
        fin = np.isfinite(vals)
        back = ora.encode_f32(vals[fin].astype(np.float32), name)
        if not np.array_equal(back, allbits[fin]):
            bad = np.nonzero(back != allbits[fin])[0][:4]
            raise AssertionError(f"{name}: round trip differs at {allbits[fin][bad]}")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        [6.0e4, 6.6e4, 7.0e4, -1e-7, 3e-8, 2.98e-8, 0.0, -0.0]]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref16 = x.astype(np.float16).view(np.uint16)
    if not np.array_equal(ora.encode_f32(x, "f16"), ref16):
        raise AssertionError("f16 encoder differs from numpy's float16 cast")
    refbf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if not np.array_equal(ora.encode_f32(x, "bf16"), refbf):
        raise AssertionError("bf16 encoder differs from torch's bfloat16 cast")
    a = np.arange(0x3c00, 0x3c40, dtype=np.uint16)  # consecutive fp16 values in [1, 2)
    av = ora.decode_bits(a, "f16")
    mid = ((av[:-1] + av[1:]) / 2).astype(np.float32)  # exact in fp32
    want = np.where(a[:-1] % 2 == 0, a[:-1], a[1:])
    if not np.array_equal(ora.encode_f32(mid, "f16"), want):
        raise AssertionError("fp16 ties are not broken to even")
    a = np.arange(0x3f80, 0x3fc0, dtype=np.uint16)  # consecutive bf16 values in [1, 2)
    av = ora.decode_bits(a, "bf16")
    mid = ((av[:-1] + av[1:]) / 2).astype(np.float32)
    want = np.where(a[:-1] % 2 == 0, a[:-1], a[1:])
    if not np.array_equal(ora.encode_f32(mid, "bf16"), want):
        raise AssertionError("bf16 ties are not broken to even")


def _rope_fp64(x64, c, s):
    """The rotation in float64 on decoded values: x*cos + rotate_half(x)*sin."""
    half = x64.shape[-1] // 2
    rot = np.concatenate([-x64[..., half:], x64[..., :half]], axis=-1)
    return x64 * c + rot * s


def pin_rope_identity_and_quarter_turn(ora):
    """cos = 1, sin = 0 leaves every bit in place; cos = 0, sin = 1 is
    rotate_half exactly: [-x[D/2:], x[:D/2]] (a sign flip and a swap of the
    halves, no rounding)."""
    for dtype in ("f16", "bf16"):
        for D in (64, 128):
            x = _bits(W.randn((3, 4, D), dtype, W.generator(D)))
            pos = np.array([0, 2, 1], np.int32)
            one, zero = np.ones((3, D), np.float32), np.zeros((3, D), np.float32)
            got, bad = ora.rope(x, one, zero, pos, dtype)
            if bad or not np.array_equal(got, x):
                raise AssertionError(f"{dtype} D{D}: identity rotation changed bits")
            got, _ = ora.rope(x, zero, one, pos, dtype)
            half = D // 2
            want = np.concatenate([x[..., half:] ^ np.uint16(0x8000), x[..., :half]], axis=-1)
            if not np.array_equal(got, want):
                raise AssertionError(f"{dtype} D{D}: quarter turn is not rotate_half")


def pin_rope_within_one_rounding_of_exact(ora):
    """Random angles: the oracle's fp32 evaluation rounded to the storage
    type lies within one unit in the last place of the exact rotation."""
    for dtype, ulp_rel in (("f16", 2.0 ** -10), ("bf16", 2.0 ** -7)):
        D = 128
        c, s = W.random_rope_tables(16, D, seed=3)
        xt = W.randn((4, 8, D), dtype, W.generator(4))
        pos = np.array([0, 5, 15, 9], np.int32)
        got, _ = ora.rope(_bits(xt), c.numpy(), s.numpy(), pos, dtype)
        exact = _rope_fp64(_exact_f64(xt), c.numpy().astype(np.float64)[pos][:, None, :],
                           s.numpy().astype(np.float64)[pos][:, None, :])
        g = ora.decode_bits(got, dtype)
        err = np.abs(g - exact)
        tol = ulp_rel * np.maximum(np.abs(exact), 2.0 ** -14) * 1.01
        if not np.all(err <= tol):
            i = np.argmax(err / tol)
            raise AssertionError(f"{dtype}: rotation off by {err.flat[i]:.3g} (tol {tol.flat[i]:.3g})")


def pin_rope_preserves_pair_norms(ora):
    """A rotation keeps the length of every (x[i], x[i + D/2]) pair."""
    D = 64
    c, s = W.random_rope_tables(8, D, seed=6)
    xt = W.randn((2, 16, D), "f16", W.generator(7))
    pos = np.array([3, 7], np.int32)
    got, _ = ora.rope(_bits(xt), c.numpy(), s.numpy(), pos, "f16")
    x = _exact_f64(xt)
    g = ora.decode_bits(got, "f16")
    n0 = x[..., :D // 2] ** 2 + x[..., D // 2:] ** 2
    n1 = g[..., :D // 2] ** 2 + g[..., D // 2:] ** 2
    if not np.allclose(n1, n0, rtol=4e-3, atol=1e-6):
        raise AssertionError("pair norms not preserved")


def pin_rope_scores_depend_on_relative_position(ora):
    """With the frequency-ladder tables, <rope(q, m), rope(k, n)> depends only
    on m - n: shifting both positions by the same amount keeps the score
    (within the rounding of the stored vectors)."""
    D = 128
    c, s = W.rope_tables(600, D)
    q = W.randn((1, 1, D), "f16", W.generator(8))
    k = W.randn((1, 1, D), "f16", W.generator(9))

    def score(m, n):
        rq, _ = ora.rope(_bits(q), c.numpy(), s.numpy(), np.array([m], np.int32), "f16")
        rk, _ = ora.rope(_bits(k), c.numpy(), s.numpy(), np.array([n], np.int32), "f16")
        return float(np.dot(ora.decode_bits(rq, "f16").ravel(), ora.decode_bits(rk, "f16").ravel()))

    scale = float(np.linalg.norm(_exact_f64(q)) * np.linalg.norm(_exact_f64(k)))
    for m, n, t in ((10, 3, 200), (0, 0, 517), (250, 249, 300)):
        a, b = score(m, n), score(m + t, n + t)
        if abs(a - b) > 4e-3 * scale:
            raise AssertionError(f"score({m},{n})={a} vs score({m + t},{n + t})={b}")
    # and it does change with the distance
    if abs(score(10, 3) - score(10, 9)) < 1e-3 * scale:
        raise AssertionError("scores ignore the relative position")


def pin_rope_position_bounds(ora):
    """A position outside the tables is counted and its rows left untouched."""
    D = 64
    c, s = W.rope_tables(10, D)
    x = _bits(W.randn((3, 2, D), "bf16", W.generator(10)))
    got, bad = ora.rope(x, c.numpy(), s.numpy(), np.array([10, 4, -1], np.int32), "bf16")
    if bad != 2 or np.any(got[0]) or np.any(got[2]) or not np.any(got[1]):
        raise AssertionError("out-of-range positions not reported")


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(ora) -> dict:
    results = {}
    for pin in PINS:
        try:
            pin(ora)
            results[pin.__name__] = "ok"
        except Exception as e:  # noqa: BLE001 - report every failure by name
            results[pin.__name__] = f"{type(e).__name__}: {e}"
    return results


if __name__ == "__main__":
    import oracle

    lib = sys.argv[1] if len(sys.argv) > 1 else None
    print(json.dumps(run_all(oracle.Oracle(lib))))
