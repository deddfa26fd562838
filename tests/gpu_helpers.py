"""Helpers shared by the GPU parity tests: run a decode step through the
CUDA library (C ABI via the binding) and the same step through the oracle,
and compare them under the tolerances of the method."""
from __future__ import annotations

import os

import numpy as np
import torch

import decode_attention_static_gb300 as da
import workloads as W

# fp16/bf16 inputs with fp32 accumulation against the fp64 oracle.
REL_FROB_TOL = 5e-3
MAX_ABS_TOL = 2e-2
THREADS = max(1, min(16, os.cpu_count() or 1))


def bits(t: torch.Tensor) -> np.ndarray:
    return W.raw_bits(t)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "") -> dict:
    g = gpu.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    assert np.all(np.isfinite(ref)), f"{what}: non-finite oracle output"
    diff = g - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    mabs = float(np.abs(diff).max()) if diff.size else 0.0
    assert rel <= REL_FROB_TOL, f"{what}: rel-Frobenius {rel:.3e} > {REL_FROB_TOL}"
    assert mabs <= MAX_ABS_TOL, f"{what}: max-abs {mabs:.3e} > {MAX_ABS_TOL}"
    return {"rel_frob": rel, "max_abs": mabs}


def oracle_step(ora, step: W.DecodeStep):
    """The oracle's append on copies of the cache bits, then its attention.
    Returns (k_bits, v_bits, out_f64)."""
    kb, vb = bits(step.k_cache).copy(), bits(step.v_cache).copy()
    ora.kvcache_append(kb, vb, bits(step.k_new), bits(step.v_new), step.position_ids.numpy())
    out = ora.decode_attn(bits(step.q), kb, vb, step.kv_len.numpy(), step.n_head, step.n_kv_head, step.dtype,
                          threads=THREADS)
    return kb, vb, out


def gpu_step(step: W.DecodeStep, fused: bool, hint: int = 0, stream_check: bool = True):
    """Append + attend on the GPU; returns (device step, out, err flag value)."""
    d = step.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fused:
        out = da.decode_step_fwd(d.q, d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids,
                                 max_kv_len_hint=hint, err_flag=err)
    else:
        da.kvcache_append(d.k_cache, d.v_cache, d.k_new, d.v_new, d.position_ids, err_flag=err)
        out = da.decode_attn_fwd(d.q, d.k_cache, d.v_cache, d.kv_len.contiguous(), max_kv_len_hint=hint,
                                 err_flag=err)
    torch.cuda.synchronize()
    return d, out, int(err.item())


def check_step(ora, step: W.DecodeStep, fused: bool, hint: int = 0, what: str = "") -> dict:
    kb, vb, ref = oracle_step(ora, step)
    d, out, err = gpu_step(step, fused, hint)
    assert err == 0, f"{what}: device error flag {err}"
    assert np.array_equal(bits(d.k_cache), kb), f"{what}: K cache differs from the oracle's append"
    assert np.array_equal(bits(d.v_cache), vb), f"{what}: V cache differs from the oracle's append"
    return assert_close(out, ref, what)
