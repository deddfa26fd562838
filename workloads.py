"""Seeded synthetic inputs for decode attention over a static KV cache.

This module only draws and lays out inputs; it holds none of the attention
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws standard-normal fp32 values, which are rounded to the storage
dtype (fp16 or bf16). Cache rows at or beyond a sequence's active length are
filled with the canonical quiet NaN of the dtype, so that any read past the
active prefix poisons the result. Draw order is fixed: q, the K cache prefix,
the V cache prefix, k_new, v_new.

Workload shapes (all q_len = 1, caches laid out [B, n_kv_head, capacity, D]):
  * tiny GQA decode: B=1, 4 query heads on 1 KV head, D=64, capacity 256,
    fp16; one append at position 36, then attention over 37 rows.
  * MHA decode sweep: B=1, 16 query and 16 KV heads, D=128, fp16,
    kv_len in {1024, 4096, 8192}, capacity = kv_len.
  * S2-Pro-shaped generation: 36 layers, 32 query / 8 KV heads, D=128, bf16,
    capacity 32768; a 234-row prompt prefix then 400 decode steps (kv_len
    235..634), append then attend in every layer at every step.
  * long-context decode: B=1, 32 query / 8 KV heads, D=128, bf16, capacity =
    kv_len = 32768.
  * batched streaming decode: B=8, 16 query / 8 KV heads, D=128, bf16,
    capacity 8192; position_id per sequence uniform in [0, 8191] with
    sequence 3 forced to position 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
# Canonical quiet NaN bit patterns.
NAN_BITS = {torch.float16: 0x7E00, torch.bfloat16: 0x7FC0}


def torch_dtype(dtype) -> torch.dtype:
    if isinstance(dtype, torch.dtype):
        return dtype
    return DTYPES[dtype]


def dtype_name(dtype) -> str:
    dt = torch_dtype(dtype)
    return "f16" if dt == torch.float16 else "bf16"


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn(shape, dtype, gen: torch.Generator) -> torch.Tensor:
    """Standard-normal fp32 draws rounded to ``dtype`` (CPU)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch_dtype(dtype))


def nan_like(shape, dtype, device="cpu") -> torch.Tensor:
    """A tensor of the dtype's canonical quiet NaN."""
    dt = torch_dtype(dtype)
    return torch.full(shape, NAN_BITS[dt], dtype=torch.int16, device=device).view(dt)


def raw_bits(t: torch.Tensor):
    """The uint16 storage of a 16-bit tensor as a numpy array (CPU copy)."""
    import numpy as np

    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16)


@dataclass
class DecodeStep:
    """Inputs of one append + attend step.

    q [B, n_head, D]; k_cache/v_cache [B, n_kv_head, capacity, D] with rows
    >= position_ids[b] NaN (the append writes row position_ids[b]); k_new and
    v_new [B, n_kv_head, D]; position_ids int32 [B]; kv_len = position_ids + 1.
    """

    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    position_ids: torch.Tensor
    n_head: int
    n_kv_head: int
    dtype: str
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def capacity(self) -> int:
        return self.k_cache.shape[2]

    @property
    def kv_len(self) -> torch.Tensor:
        return (self.position_ids + 1).to(torch.int32)

    def to(self, device) -> "DecodeStep":
        return DecodeStep(self.q.to(device), self.k_cache.to(device), self.v_cache.to(device),
                          self.k_new.to(device), self.v_new.to(device), self.position_ids.to(device),
                          self.n_head, self.n_kv_head, self.dtype, dict(self.meta))


def cache_prefix(B: int, n_kv_head: int, rows: int, head_dim: int, dtype, filled, gen) -> torch.Tensor:
    """[B, n_kv_head, rows, D] with rows >= filled[b] set to NaN."""
    t = randn((B, n_kv_head, rows, head_dim), dtype, gen)
    for b in range(B):
        f = int(filled[b])
        if f < rows:
            t[b, :, f:, :] = nan_like((n_kv_head, rows - f, head_dim), dtype)
    return t


def decode_step(B: int, n_head: int, n_kv_head: int, head_dim: int, capacity: int, dtype,
                position_ids, seed: int = 0) -> DecodeStep:
    """One append + attend step: cache rows [0, position_ids[b]) random,
    the rest NaN; new rows and q random. CPU tensors."""
    pos = torch.as_tensor(position_ids, dtype=torch.int32).reshape(B)
    gen = generator(seed)
    q = randn((B, n_head, head_dim), dtype, gen)
    k_cache = cache_prefix(B, n_kv_head, capacity, head_dim, dtype, pos.tolist(), gen)
    v_cache = cache_prefix(B, n_kv_head, capacity, head_dim, dtype, pos.tolist(), gen)
    k_new = randn((B, n_kv_head, head_dim), dtype, gen)
    v_new = randn((B, n_kv_head, head_dim), dtype, gen)
    return DecodeStep(q, k_cache, v_cache, k_new, v_new, pos, n_head, n_kv_head, dtype_name(dtype),
                      {"seed": seed})


# ---------------------------------------------------------------------------
# The named workloads.

def tiny_gqa(seed: int = 0) -> DecodeStep:
    """B=1, 4 query heads / 1 KV head, D=64, capacity 256, fp16, append at 36."""
    s = decode_step(1, 4, 1, 64, 256, "f16", [36], seed)
    s.meta["workload"] = "tiny GQA decode"
    return s


MHA_SWEEP_KV_LENS = (1024, 4096, 8192)


def mha_sweep(kv_len: int, seed: int = 0, extra_capacity: int = 0) -> DecodeStep:
    """B=1, 16 query and 16 KV heads, D=128, fp16, capacity = kv_len (plus an
    optional NaN tail of ``extra_capacity`` rows); append at kv_len - 1."""
    s = decode_step(1, 16, 16, 128, kv_len + extra_capacity, "f16", [kv_len - 1], seed)
    s.meta["workload"] = f"MHA decode sweep kv_len {kv_len}"
    return s


def long_context(seed: int = 0, kv_len: int = 32768, capacity: int = 32768) -> DecodeStep:
    """B=1, 32 query / 8 KV heads, D=128, bf16, full 32768-row cache."""
    s = decode_step(1, 32, 8, 128, capacity, "bf16", [kv_len - 1], seed)
    s.meta["workload"] = f"long-context decode kv_len {kv_len}"
    return s


def batched_positions(seed: int = 0, B: int = 8, capacity: int = 8192, zero_at: int = 3) -> torch.Tensor:
    """position_id per sequence, uniform in [0, capacity - 1], one forced to 0."""
    gen = generator(seed + 7919)
    pos = torch.randint(0, capacity, (B,), generator=gen, dtype=torch.int64).to(torch.int32)
    if 0 <= zero_at < B:
        pos[zero_at] = 0
    return pos


def batched_streaming(seed: int = 0) -> DecodeStep:
    """B=8, 16 query / 8 KV heads, D=128, bf16, capacity 8192, ragged positions."""
    pos = batched_positions(seed)
    s = decode_step(8, 16, 8, 128, 8192, "bf16", pos, seed)
    s.meta["workload"] = "batched streaming decode"
    return s


@dataclass
class Generation:
    """S2-Pro-shaped multi-layer generation inputs (CPU tensors).

    k_prefix/v_prefix [layers, B, n_kv_head, prompt, D]: the prompt rows of
    every layer's cache. q [steps, layers, B, n_head, D]; k_new/v_new
    [steps, layers, B, n_kv_head, D]. Step i appends at prompt + i and
    attends over prompt + i + 1 rows.
    """

    layers: int
    B: int
    n_head: int
    n_kv_head: int
    head_dim: int
    capacity: int
    prompt: int
    steps: int
    dtype: str
    k_prefix: torch.Tensor
    v_prefix: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor

    def position(self, step: int) -> int:
        return self.prompt + step


def s2pro_generation(seed: int = 0, layers: int = 36, prompt: int = 234, steps: int = 400,
                     capacity: int = 32768) -> Generation:
    """36 layers, 32 query / 8 KV heads, D=128, bf16, capacity 32768, prompt
    234, 400 decode steps (kv_len 235..634)."""
    B, H, Hkv, D, dt = 1, 32, 8, 128, "bf16"
    gen = generator(seed)
    q = randn((steps, layers, B, H, D), dt, gen)
    k_prefix = randn((layers, B, Hkv, prompt, D), dt, gen)
    v_prefix = randn((layers, B, Hkv, prompt, D), dt, gen)
    k_new = randn((steps, layers, B, Hkv, D), dt, gen)
    v_new = randn((steps, layers, B, Hkv, D), dt, gen)
    return Generation(layers, B, H, Hkv, D, capacity, prompt, steps, dt, k_prefix, v_prefix, q,
                      k_new, v_new)


def rope_tables(rows: int, head_dim: int, base: float = 10000.0) -> tuple[torch.Tensor, torch.Tensor]:
    """Position-embedding tables of the usual rotary scheme, as a model hands
    them to its attention: row p holds cos(p * w_i) and sin(p * w_i) for the
    frequencies w_i = base^(-2i / head_dim), i < head_dim / 2, repeated for the
    two halves of the head ([rows, head_dim] fp32, computed in fp64). Model
    parameters and inputs, not the method's arithmetic."""
    half = head_dim // 2
    w = base ** (-torch.arange(half, dtype=torch.float64) * 2.0 / head_dim)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * w[None, :]
    ang = torch.cat([ang, ang], dim=1)
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


def random_rope_tables(rows: int, head_dim: int, seed: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Tables with a random angle per (row, frequency), halves repeated: for
    tests that want every rotation, not one frequency ladder."""
    gen = generator(seed)
    ang = torch.rand((rows, head_dim // 2), generator=gen, dtype=torch.float64) * (2 * torch.pi) - torch.pi
    ang = torch.cat([ang, ang], dim=1)
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)
