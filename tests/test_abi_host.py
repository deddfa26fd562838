"""The C ABI on the host: the library loads, exports every symbol the header
declares, and rejects bad arguments before touching the GPU (CPU only; no
compute call is made)."""
import ctypes
import pathlib
import re
import subprocess

import pytest
import torch

import decode_attention_static_gb300 as da
from decode_attention_static_gb300 import build as da_build

ROOT = pathlib.Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    da_build.build_library()
    return da.load_library()


def declared_symbols():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = h.read_text()
        names |= set(re.findall(r"^DA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_entry_points():
    names = declared_symbols()
    assert {"kvcache_append", "decode_attn_fwd", "decode_step_fwd", "decode_attn_workspace_size",
            "decode_attn_plan_splits", "da_status_string", "da_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(da.library_path())], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared_symbols() - exported
    assert not missing, f"declared but not exported: {missing}"
    for name in declared_symbols():
        assert getattr(lib, name) is not None
    assert declared_symbols() <= set(da.exported_symbols()), "binding lacks a declared entry point"


def test_status_strings(lib):
    for code in range(-7, 1):
        assert da.status_string(code) not in ("", "unknown status")
    assert da.status_string(-99) == "unknown status"


def test_plan_splits_properties(lib):
    sms, per = 152, 3
    # one (b, kv-head) group per CTA already fills the GPU: no split
    assert da.plan_splits(64, 8, 128, 32768, sms, per) == (1, 1)
    # short prefix (16 tiles of 64 rows): one cluster per group, at most one
    # CTA per SM (152 // 16 = 9) and about `per` tiles per CTA (16 / 3 -> 6)
    assert da.plan_splits(1, 16, 128, 1024, sms, per) == (6, 6)
    # long prefix of one sequence whose largest clusters cover every SM
    # (16 groups x 16 >= 152): one cluster per group, merged on chip
    assert da.plan_splits(1, 16, 128, 8192, sms, per) == (16, 16)
    # long prefix whose clusters would leave SMs idle (8 x 16 < 152): every
    # resident CTA streams rows, merged through the workspace
    assert da.plan_splits(1, 8, 128, 32768, sms, per) == (57, 1)
    # one CTA per SM (four query heads per KV head): a split may stream up to
    # 8 tiles and still be served by one cluster per group
    assert da.plan_splits(1, 8, 128, 4096, sms, 1, cluster_max=12) == (12, 12)
    assert da.plan_splits(1, 8, 128, 6144, sms, 1, cluster_max=12) == (12, 12)
    assert da.plan_splits(1, 8, 128, 8192, sms, 1, cluster_max=12) == (19, 1)
    assert da.plan_splits(1, 8, 128, 4096, sms, per, cluster_max=12) == (57, 1)
    # a batch: two waves' worth of splits (most sequences are shorter than the bound)
    assert da.plan_splits(8, 8, 128, 8192, sms, per) == (14, 1)
    # without clusters a short prefix is split flat too
    assert da.plan_splits(1, 16, 128, 1024, sms, per, cluster_max=1) == (16, 1)
    # never more splits than tiles (64 rows at D=128, 128 at D=64); two tiles
    # are too short to share between CTAs holding `per` tiles each
    assert da.plan_splits(1, 1, 128, 100, sms, per) == (1, 1)
    assert da.plan_splits(1, 1, 128, 100, sms, 1) == (2, 2)
    assert da.plan_splits(1, 1, 64, 100, sms, per) == (1, 1)
    assert da.plan_splits(1, 1, 128, 1, sms, per) == (1, 1)
    # splits are whole clusters, fit one wave, and never shrink as the bound grows,
    # so a workspace sized for the capacity fits any hint
    for B, Hkv in [(1, 8), (1, 16), (2, 8), (8, 8), (4, 2), (3, 5)]:
        prev = 0
        for n in range(1, 40000, 397):
            s, cs = da.plan_splits(B, Hkv, 128, n, sms, per)
            assert s % cs == 0 and s >= prev and 1 <= cs <= 16
            assert s == 1 or s * B * Hkv <= sms * per * (2 if B > 1 else 1)
            prev = s
    for bad in [(0, 8, 128, 10, sms, per, 16), (1, 0, 128, 10, sms, per, 16), (1, 8, 128, 0, sms, per, 16),
                (1, 8, 128, 10, 0, per, 16), (1, 8, 128, 10, sms, 0, 16), (1, 8, 128, 10, sms, per, 0)]:
        assert lib.decode_attn_plan_splits(*bad, None) == -2
    assert lib.decode_attn_plan_splits(1, 8, 96, 10, sms, per, 16, None) == -3


A = 0x10000  # a 16-byte-aligned address that is never dereferenced by these calls


def _fwd(lib, **kw):
    args = dict(q=A, k=A, v=A, kv_len=A, B=1, H=32, Hkv=8, D=128, cap=1024, scale=0.1, out=A, ws=A, ws_bytes=1 << 30,
                hint=0, dtype=1, err=None, stream=None)
    args.update(kw)
    return lib.decode_attn_fwd(args["q"], args["k"], args["v"], args["kv_len"], args["B"], args["H"], args["Hkv"],
                               args["D"], args["cap"], args["scale"], args["out"], args["ws"], args["ws_bytes"],
                               args["hint"], args["dtype"], args["err"], args["stream"])


def test_decode_attn_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, dtype=2) == -7
    assert _fwd(lib, dtype=-1) == -7
    assert _fwd(lib, H=30) == -2          # n_head not a multiple of n_kv_head
    assert _fwd(lib, B=-1) == -2
    assert _fwd(lib, cap=0) == -2
    assert _fwd(lib, Hkv=0) == -2
    assert _fwd(lib, B=70000) == -2
    assert _fwd(lib, D=96) == -3
    assert _fwd(lib, D=256) == -3
    assert _fwd(lib, H=24, Hkv=8) == -3   # group 3 not built
    assert _fwd(lib, H=128, Hkv=8) == -3  # group 16 not built
    assert _fwd(lib, q=None) == -1
    assert _fwd(lib, kv_len=None) == -1
    assert _fwd(lib, out=None) == -1
    assert _fwd(lib, q=A + 8) == -6
    assert _fwd(lib, out=A + 2) == -6
    assert _fwd(lib, B=0, q=None, k=None) == 0  # empty batch: nothing to do


def test_decode_step_and_append_reject_bad_arguments(lib):
    st = lib.decode_step_fwd(A, A, A, None, A, A, 1, 32, 8, 128, 1024, 0.1, A, A, 1 << 30, 0, 1, None, None)
    assert st == -1
    st = lib.decode_step_fwd(A, A, A, A, A + 4, A, 1, 32, 8, 128, 1024, 0.1, A, A, 1 << 30, 0, 1, None, None)
    assert st == -6
    assert lib.kvcache_append(A, A, A, A, A, 1, 8, 128, 1024, 5, None, None) == -7
    assert lib.kvcache_append(A, A, A, A, A, 1, 8, 12, 1024, 1, None, None) == -2
    assert lib.kvcache_append(A, A, A, A, A, 1, 8, 128, 0, 1, None, None) == -2
    assert lib.kvcache_append(A, None, A, A, A, 1, 8, 128, 1024, 1, None, None) == -1
    assert lib.kvcache_append(A, A, A + 1, A, A, 1, 8, 128, 1024, 1, None, None) == -6
    assert lib.kvcache_append(None, None, None, None, None, 0, 8, 128, 1024, 1, None, None) == 0


def test_decode_step_layers_rejects_bad_arguments(lib):
    def layers_call(layers=2, k_new=A, D=128, B=1):
        return lib.decode_step_layers_fwd(A, A, A, k_new, A, A, layers, B, 32, 8, D, 1024, 0.1, A, A, 1 << 30, 0, 1,
                                          None, None)

    assert layers_call(layers=-1) == -2
    assert layers_call(layers=0) == 0
    assert layers_call(k_new=None) == -1
    assert layers_call(D=96) == -3
    assert layers_call(k_new=A + 4) == -6
    # the stack is one batch of layers * B sequences (the grid's z extent)
    assert layers_call(layers=300, B=300) == -2


def test_decode_step_rope_rejects_bad_tables(lib):
    def rope(cos=A, sin=A, rows=1024, cap=1024):
        return lib.decode_step_rope_fwd(A, A, A, A, A, cos, sin, rows, A, 1, 32, 8, 128, cap, 0.1, A, A, 1 << 30, 0, 1,
                                        None, None)

    assert rope(cos=None) == -1
    assert rope(sin=None) == -1
    assert rope(rows=1023) == -2          # every valid position needs a table row
    assert rope(cos=A + 4) == -6
    assert rope(sin=A + 8) == -6


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert _fwd(lib) == -5
    assert lib.decode_attn_workspace_size(1, 32, 8, 128, 1024) == ctypes.c_size_t(-1).value


def test_kernel_for_rejects_bad_sizes_without_a_device(lib):
    # validated before any device query: group size, head_dim, dtype
    assert lib.decode_attn_kernel_for(1, 30, 8, 128, 1024, 0, 1, 0) == -2   # n_head % n_kv_head
    assert lib.decode_attn_kernel_for(1, 32, 8, 96, 1024, 0, 1, 0) == -3    # unsupported head_dim
    assert lib.decode_attn_kernel_for(1, 48, 4, 128, 1024, 0, 1, 0) == -3   # unsupported group size 12
    assert lib.decode_attn_kernel_for(1, 32, 8, 128, 1024, 0, 7, 0) == -7   # unknown dtype
    assert lib.decode_attn_kernel_for(0, 32, 8, 128, 1024, 0, 1, 0) == 0    # empty batch: nothing launched


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.decode_attn_workspace_size(1, 30, 8, 128, 1024) == ctypes.c_size_t(-1).value
    assert lib.decode_attn_workspace_size(1, 32, 8, 100, 1024) == ctypes.c_size_t(-1).value
    assert lib.decode_attn_workspace_size(0, 32, 8, 128, 1024) == 0


def test_binding_checks_tensor_arguments():
    cpu = torch.zeros(1, 4, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        da.decode_attn_fwd(cpu, torch.zeros(1, 1, 8, 64, dtype=torch.float16),
                           torch.zeros(1, 1, 8, 64, dtype=torch.float16), torch.ones(1, dtype=torch.int32))


def test_plain_c_program_uses_the_library(lib, tmp_path):
    """The boundary is a C ABI: the header compiles as C99, and a plain C
    program links against the library and calls host-only entry points."""
    src = tmp_path / "consumer.c"
    src.write_text(
        '#include <stdio.h>\n#include <string.h>\n#include "decode_attn.h"\n'
        "int main(void) {\n"
        "  int cs = 0;\n"
        "  int s = decode_attn_plan_splits(1, 16, 128, 8192, 152, 2, 16, &cs);\n"
        '  if (da_version() <= 0 || strcmp(da_status_string(DA_OK), "") == 0) return 1;\n'
        "  if (decode_attn_plan_splits(0, 16, 128, 8192, 152, 2, 16, &cs) != DA_ERR_SHAPE) return 2;\n"
        "  int kv0, nkv, h0, nh;\n"
        "  if (decode_attn_shard_heads(32, 8, 3, 2, &kv0, &nkv, &h0, &nh) != DA_OK) return 4;\n"
        "  if (kv0 != 6 || nkv != 2 || h0 != 24 || nh != 8) return 5;\n"
        '  printf("%d %d\\n", s, cs);\n'
        "  return s >= 1 && cs >= 1 ? 0 : 3;\n}\n")
    exe = tmp_path / "consumer"
    libdir = da.library_path().parent
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", str(src), f"-I{ROOT / 'include'}",
                    f"-L{libdir}", f"-l:{da.library_path().name}", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert (int(out[0]), int(out[1])) == da.plan_splits(1, 16, 128, 8192, 152, 2)


@pytest.mark.parametrize("entry", ["decode_attn_fwd", "decode_step_fwd", "decode_step_rope_fwd",
                                   "decode_step_layers_fwd", "kvcache_append", "decode_attn_fwd_static_scratch"])
def test_binding_rejects_host_tensors_before_any_call(entry):
    """Every binding entry point checks its tensors (device, contiguity) before
    it reaches the library: host tensors raise ValueError, nothing runs."""
    f16 = torch.float16
    q = torch.zeros(1, 4, 64, dtype=f16)
    kc = torch.zeros(1, 1, 8, 64, dtype=f16)
    kn = torch.zeros(1, 1, 64, dtype=f16)
    pos = torch.zeros(1, dtype=torch.int32)
    calls = {
        "decode_attn_fwd": lambda: da.decode_attn_fwd(q, kc, kc, pos),
        "decode_step_fwd": lambda: da.decode_step_fwd(q, kc, kc, kn, kn, pos),
        "decode_step_rope_fwd": lambda: da.decode_step_rope_fwd(q, kc, kc, kn, kn, torch.zeros(8, 64),
                                                                torch.zeros(8, 64), pos),
        "decode_step_layers_fwd": lambda: da.decode_step_layers_fwd(q[None], kc[None], kc[None], kn[None], kn[None],
                                                                    pos),
        "kvcache_append": lambda: da.kvcache_append(kc, kc, kn, kn, pos),
        "decode_attn_fwd_static_scratch": lambda: da.decode_attn_fwd_static_scratch(q, kc, kc, pos),
    }
    with pytest.raises(ValueError):
        calls[entry]()


def test_prefix_ready_blocks_nest_and_restore(lib):
    """The binding's prefix_ready() block restores the thread's previous
    setting (host-side state only; no GPU call)."""
    from decode_attention_static_gb300 import _binding as B

    da.set_prefix_ready(False)
    with da.prefix_ready():
        assert B._thread_state.prefix_ready
        with da.prefix_ready():
            assert B._thread_state.prefix_ready
        assert B._thread_state.prefix_ready
    assert not B._thread_state.prefix_ready
