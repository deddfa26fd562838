"""ctypes binding of libdecode_attn.so: argument marshalling only.

Every function here takes torch tensors that already live on the GPU, checks
that their shapes agree, and passes raw pointers, sizes and the current CUDA
stream to the C entry point of the same name. All computation happens in the
library's kernels. If the library has not been built, every call raises
``LibraryNotBuilt`` — there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import pathlib
import threading

import torch

LIBRARY = pathlib.Path(__file__).resolve().parent / "libdecode_attn.so"

DA_F16 = 0
DA_BF16 = 1
DA_DEVERR_KV_LEN = 1
DA_DEVERR_POSITION = 2
DA_DEVERR_TIMEOUT = 4
DA_DEVERR_WORKSPACE = 8

_DTYPE_CODE = {torch.float16: DA_F16, torch.bfloat16: DA_BF16}


class LibraryNotBuilt(RuntimeError):
    pass


class DecodeAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_SIGNATURES = {
    "da_status_string": ([_i], ctypes.c_char_p),
    "da_version": ([], _i),
    "decode_attn_plan_splits": ([_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i)], _i),
    "decode_attn_workspace_size": ([_i, _i, _i, _i, _i], ctypes.c_size_t),
    "decode_attn_workspace_init": ([_vp, ctypes.c_size_t, _vp], _i),
    "decode_attn_splits_for": ([_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i)], _i),
    "decode_attn_kernel_for": ([_i, _i, _i, _i, _i, _i, _i, _i], _i),
    "da_set_timing_events": ([_vp, _vp], _i),
    "kvcache_append": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "decode_attn_fwd": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp, ctypes.c_size_t, _i, _i,
                         _vp, _vp], _i),
    "decode_attn_fwd_static_scratch": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _i, _i, _vp,
                                        _vp], _i),
    "decode_step_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp, ctypes.c_size_t,
                         _i, _i, _vp, _vp], _i),
    "da_test_skip_slot": ([_i], _i),
    "da_set_prefix_ready": ([_i], _i),
    "decode_attn_shard_heads": ([_i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i),
                                 ctypes.POINTER(_i)], _i),
    "decode_step_layers_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp,
                                ctypes.c_size_t, _i, _i, _vp, _vp], _i),
    "decode_step_rope_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp,
                              ctypes.c_size_t, _i, _i, _vp, _vp], _i),
}


def library_path() -> pathlib.Path:
    return LIBRARY


def load_library() -> ctypes.CDLL:
    """Load the CUDA library (once). Raises LibraryNotBuilt if it is missing."""
    global _lib
    if _lib is None:
        if not LIBRARY.exists():
            raise LibraryNotBuilt(f"{LIBRARY} is missing: build it with decode_attention_static_gb300.build")
        lib = ctypes.CDLL(str(LIBRARY))
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def status_string(status: int) -> str:
    return load_library().da_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise DecodeAttnError(fn, status, status_string(status))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


# Fast accessors of torch's current device and raw current stream (plain
# integers, no Python objects), with the public API as the fallback.
_raw_stream_of = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_current_device_index = getattr(torch._C, "_cuda_getDevice", None)


def _raw_stream(index: int) -> int:
    if _raw_stream_of is not None:
        return _raw_stream_of(index)
    return torch.cuda.current_stream(index).cuda_stream


def _device_now() -> int:
    return _current_device_index() if _current_device_index is not None else torch.cuda.current_device()


def _same_device_contiguous(index: int, names: tuple, tensors: tuple) -> None:
    """Every tensor is a contiguous CUDA tensor on device `index` (one pass;
    the detailed check runs only to name the offending tensor)."""
    for name, t in zip(names, tensors):
        if t.get_device() != index or not t.is_contiguous():
            _on(torch.device("cuda", index), **{name: t})
            raise ValueError(f"{name} must be a contiguous CUDA tensor on cuda:{index}")


def _call_on(fn: str, index: int, *args) -> None:
    """_call for a device given by index."""
    f = getattr(load_library(), fn)
    if _device_now() == index:
        st = f(*args)
    else:
        with torch.cuda.device(index):
            st = f(*args)
    if st != 0:
        _check(fn, st)


def _code_for(dtype: torch.dtype) -> int:
    if dtype not in _DTYPE_CODE:
        raise TypeError(f"dtype {dtype} is not supported (float16 or bfloat16)")
    return _DTYPE_CODE[dtype]


def _dtype_code(t: torch.Tensor) -> int:
    return _code_for(t.dtype)


def _require(cond: bool, msg) -> None:
    """Raise ValueError(msg) unless cond; msg may be a callable giving the
    message (so that it is only formatted on failure)."""
    if not cond:
        raise ValueError(msg() if callable(msg) else msg)


def _cuda_contig(name: str, t: torch.Tensor) -> None:
    _require(t.is_cuda, lambda: f"{name} must be a CUDA tensor")
    _require(t.is_contiguous(), lambda: f"{name} must be contiguous")


def _on(device: torch.device, **tensors: torch.Tensor) -> None:
    """Every named tensor is a contiguous CUDA tensor on `device`."""
    for name, t in tensors.items():
        _cuda_contig(name, t)
        _require(t.device == device, lambda: f"{name} is on {t.device}, the inputs on {device}")


def _err_ptr(err_flag: torch.Tensor | None, device: torch.device):
    if err_flag is None:
        return None
    _on(device, err_flag=err_flag)
    _require(err_flag.dtype == torch.int32 and err_flag.numel() >= 1, "err_flag must be int32 with one element")
    return _ptr(err_flag)


def _workspace(workspace: torch.Tensor, device: torch.device):
    """(pointer, size in bytes) of a caller workspace."""
    _on(device, workspace=workspace)
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def _call(fn: str, device: torch.device, *args) -> None:
    """Call entry point `fn` with `device` current (the library launches on
    the current device, on the stream passed in `args`)."""
    f = getattr(load_library(), fn)
    index = device.index if device.index is not None else torch.cuda.current_device()
    if torch.cuda.current_device() == index:
        st = f(*args)
    else:
        with torch.cuda.device(device):
            st = f(*args)
    _check(fn, st)


def plan_splits(B: int, n_kv_head: int, head_dim: int, max_kv_len: int, num_sms: int, ctas_per_sm: int,
                cluster_max: int = 16) -> tuple[int, int]:
    """(splits, cluster size) of the host split plan."""
    cs = ctypes.c_int(0)
    s = load_library().decode_attn_plan_splits(B, n_kv_head, head_dim, max_kv_len, num_sms, ctas_per_sm,
                                               cluster_max, ctypes.byref(cs))
    _check("decode_attn_plan_splits", s if s < 0 else 0)
    return s, cs.value


def decode_attn_workspace_size(B: int, n_head: int, n_kv_head: int, head_dim: int, capacity: int) -> int:
    n = load_library().decode_attn_workspace_size(B, n_head, n_kv_head, head_dim, capacity)
    if n == ctypes.c_size_t(-1).value:
        raise DecodeAttnError("decode_attn_workspace_size", -2, "invalid sizes or device query failed")
    return int(n)


def alloc_workspace(B: int, n_head: int, n_kv_head: int, head_dim: int, capacity: int, device=None) -> torch.Tensor:
    """A zero-filled device byte buffer of decode_attn_workspace_size() bytes (torch owns it)."""
    n = decode_attn_workspace_size(B, n_head, n_kv_head, head_dim, capacity)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def workspace_init(workspace: torch.Tensor) -> None:
    """Zero-fill a workspace on the current stream (needed once before first use)."""
    ws, ws_bytes = _workspace(workspace, workspace.device)
    _call("decode_attn_workspace_init", workspace.device, ws, ws_bytes, _stream(workspace))


def splits_for(B: int, n_head: int, n_kv_head: int, head_dim: int, capacity: int, max_kv_len_hint: int = 0,
               dtype: torch.dtype = torch.bfloat16) -> tuple[int, int]:
    """(splits, cluster size) decode_attn_fwd will use for these sizes on the current device."""
    cs = ctypes.c_int(0)
    s = load_library().decode_attn_splits_for(B, n_head, n_kv_head, head_dim, capacity, int(max_kv_len_hint),
                                              _code_for(dtype), ctypes.byref(cs))
    _check("decode_attn_splits_for", s if s < 0 else 0)
    return s, cs.value


# decode_attn_kernel_for results
KERNEL_NAMES = {0: "cuda_cores", 1: "tensor_cores", 2: "tensor_cores_paired"}


def kernel_for(B: int, n_head: int, n_kv_head: int, head_dim: int, capacity: int, max_kv_len_hint: int = 0,
               dtype: torch.dtype = torch.bfloat16, rotary: bool = False) -> str:
    """The decode kernel a call with these sizes launches on the current device:
    "cuda_cores", "tensor_cores" or "tensor_cores_paired" (for the layers call
    pass layers * B as B)."""
    k = load_library().decode_attn_kernel_for(B, n_head, n_kv_head, head_dim, capacity, int(max_kv_len_hint),
                                              _code_for(dtype), 1 if rotary else 0)
    _check("decode_attn_kernel_for", k if k < 0 else 0)
    return KERNEL_NAMES[k]


def shard_heads(n_head: int, n_kv_head: int, world: int, rank: int) -> tuple[int, int, int, int]:
    """(kv_head0, n_kv_local, head0, n_head_local) of rank `rank` in the
    KV-head partition of decode_attn_shard_heads (host only)."""
    out = [ctypes.c_int(0) for _ in range(4)]
    st = load_library().decode_attn_shard_heads(n_head, n_kv_head, world, rank, *(ctypes.byref(o) for o in out))
    _check("decode_attn_shard_heads", st)
    return tuple(o.value for o in out)


def set_timing_events(before: "torch.cuda.Event | None", after: "torch.cuda.Event | None") -> None:
    """Record `before`/`after` around the decode kernel of every later call on
    this thread (both None turns it off). Events need timing enabled."""
    if before is None or after is None:
        load_library().da_set_timing_events(None, None)
        return
    load_library().da_set_timing_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def kvcache_append(k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   position_ids: torch.Tensor, err_flag: torch.Tensor | None = None) -> None:
    """k_cache[b, g, position_ids[b]] = k_new[b, g] (and V), in place."""
    _cuda_contig("k_cache", k_cache)
    dev = k_cache.device
    _on(dev, v_cache=v_cache, k_new=k_new, v_new=v_new, position_ids=position_ids)
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [B, n_kv_head, capacity, D]")
    B, Hkv, cap, D = k_cache.shape
    _require(tuple(k_new.shape) == (B, Hkv, D) and v_new.shape == k_new.shape, "k_new/v_new must be [B, n_kv_head, D]")
    _require(position_ids.dtype == torch.int32 and position_ids.numel() == B, "position_ids must be int32 [B]")
    _require(k_new.dtype == k_cache.dtype == v_cache.dtype == v_new.dtype, "dtypes differ")
    _call("kvcache_append", dev, _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(position_ids), B, Hkv,
          D, cap, _dtype_code(k_cache), _err_ptr(err_flag, dev), _stream(k_cache))


def _attn_shapes(q, k_cache, v_cache, out):
    _cuda_contig("q", q)
    _on(q.device, k_cache=k_cache, v_cache=v_cache, out=out)
    _require(q.dim() == 3, "q must be [B, n_head, D]")
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [B, n_kv_head, capacity, D]")
    B, H, D = q.shape
    _require(k_cache.shape[0] == B and k_cache.shape[3] == D, "cache batch/head_dim must match q")
    _require(out.shape == q.shape, "out must be [B, n_head, D]")
    _require(q.dtype == k_cache.dtype == v_cache.dtype == out.dtype, "dtypes differ")
    return B, H, k_cache.shape[1], D, k_cache.shape[2]


def decode_attn_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: torch.Tensor,
                    out: torch.Tensor | None = None, scale: float | None = None,
                    workspace: torch.Tensor | None = None, max_kv_len_hint: int = 0,
                    err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """softmax(scale * q K[:kv_len]^T) V[:kv_len] per head; returns out [B, n_head, D]."""
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("q", q)
    index = q.get_device()
    _require(q.dim() == 3, "q must be [B, n_head, D]")
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [B, n_kv_head, capacity, D]")
    B, H, D = q.shape
    _, Hkv, cap, Dk = k_cache.shape
    _require(k_cache.shape[0] == B and Dk == D, "cache batch/head_dim must match q")
    _require(out.shape == q.shape, "out must be [B, n_head, D]")
    _require(q.dtype == k_cache.dtype == v_cache.dtype == out.dtype, "dtypes differ")
    _require(kv_len.dtype == torch.int32 and kv_len.numel() == B, "kv_len must be int32 [B]")
    if workspace is None:
        workspace = alloc_workspace(B, H, Hkv, D, cap, q.device)
    names = ("k_cache", "v_cache", "out", "kv_len", "workspace")
    tensors = (k_cache, v_cache, out, kv_len, workspace)
    if err_flag is not None:
        _require(err_flag.dtype == torch.int32 and err_flag.numel() >= 1, "err_flag must be int32 with one element")
        names, tensors = names + ("err_flag",), tensors + (err_flag,)
    _same_device_contiguous(index, names, tensors)
    _call_on("decode_attn_fwd", index, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kv_len.data_ptr(), B, H,
             Hkv, D, cap, float(D ** -0.5 if scale is None else scale), out.data_ptr(), workspace.data_ptr(),
             workspace.numel() * workspace.element_size(), int(max_kv_len_hint), _code_for(q.dtype),
             None if err_flag is None else err_flag.data_ptr(), _raw_stream(index))
    return out


def _step_inputs(q, k_cache, v_cache, k_new, v_new, position_ids, out, lead=()):
    """Shapes of a fused step: q [*lead, B, H, D], caches [*lead, B, Hkv, cap, D],
    k_new/v_new [*lead, B, Hkv, D], position_ids int32 [B]."""
    n = len(lead)
    B, H, Hkv, D, cap = _attn_shapes(q[(0,) * n], k_cache[(0,) * n], v_cache[(0,) * n], out[(0,) * n])
    _on(q.device, q=q, k_cache=k_cache, v_cache=v_cache, out=out, k_new=k_new, v_new=v_new,
        position_ids=position_ids)
    _require(tuple(k_new.shape) == (*lead, B, Hkv, D) and v_new.shape == k_new.shape,
             "k_new/v_new must be [" + "layers, " * n + "B, n_kv_head, D]")
    _require(k_new.dtype == v_new.dtype == q.dtype, "dtypes differ")
    _require(position_ids.dtype == torch.int32 and position_ids.numel() == B, "position_ids must be int32 [B]")
    return B, H, Hkv, D, cap


def decode_step_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                    v_new: torch.Tensor, position_ids: torch.Tensor, out: torch.Tensor | None = None,
                    scale: float | None = None, workspace: torch.Tensor | None = None, max_kv_len_hint: int = 0,
                    err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """Fused append at position_ids then attention over [0, position_ids]."""
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("q", q)
    index = q.get_device()
    _require(q.dim() == 3, "q must be [B, n_head, D]")
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [B, n_kv_head, capacity, D]")
    B, H, D = q.shape
    _, Hkv, cap, Dk = k_cache.shape
    _require(k_cache.shape[0] == B and Dk == D, "cache batch/head_dim must match q")
    _require(out.shape == q.shape, "out must be [B, n_head, D]")
    _require(k_new.shape == (B, Hkv, D) and v_new.shape == k_new.shape, "k_new/v_new must be [B, n_kv_head, D]")
    _require(q.dtype == k_cache.dtype == v_cache.dtype == out.dtype == k_new.dtype == v_new.dtype, "dtypes differ")
    _require(position_ids.dtype == torch.int32 and position_ids.numel() == B, "position_ids must be int32 [B]")
    if workspace is None:
        workspace = alloc_workspace(B, H, Hkv, D, cap, q.device)
    names = ("k_cache", "v_cache", "out", "k_new", "v_new", "position_ids", "workspace")
    tensors = (k_cache, v_cache, out, k_new, v_new, position_ids, workspace)
    if err_flag is not None:
        _require(err_flag.dtype == torch.int32 and err_flag.numel() >= 1, "err_flag must be int32 with one element")
        names, tensors = names + ("err_flag",), tensors + (err_flag,)
    _same_device_contiguous(index, names, tensors)
    _call_on("decode_step_fwd", index, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
             v_new.data_ptr(), position_ids.data_ptr(), B, H, Hkv, D, cap, float(D ** -0.5 if scale is None else scale),
             out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
             int(max_kv_len_hint), _code_for(q.dtype), None if err_flag is None else err_flag.data_ptr(),
             _raw_stream(index))
    return out


def decode_step_rope_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                         v_new: torch.Tensor, rope_cos: torch.Tensor, rope_sin: torch.Tensor,
                         position_ids: torch.Tensor, out: torch.Tensor | None = None, scale: float | None = None,
                         workspace: torch.Tensor | None = None, max_kv_len_hint: int = 0,
                         err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """decode_step_fwd with the rotary embedding of q and k_new at
    position_ids (tables rope_cos/rope_sin fp32 [rows, D], rows >= capacity)."""
    if out is None:
        out = torch.empty_like(q)
    B, H, Hkv, D, cap = _step_inputs(q, k_cache, v_cache, k_new, v_new, position_ids, out)
    dev = q.device
    _on(dev, rope_cos=rope_cos, rope_sin=rope_sin)
    _require(rope_cos.dtype == torch.float32 and rope_sin.dtype == torch.float32 and rope_cos.dim() == 2
             and rope_cos.shape == rope_sin.shape and rope_cos.shape[1] == D, "rope tables must be fp32 [rows, D]")
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = alloc_workspace(B, H, Hkv, D, cap, dev)
    ws, ws_bytes = _workspace(workspace, dev)
    _call("decode_step_rope_fwd", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
          _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0], _ptr(position_ids), B, H, Hkv, D, cap, float(scale),
          _ptr(out), ws, ws_bytes, int(max_kv_len_hint), _dtype_code(q), _err_ptr(err_flag, dev), _stream(q))
    return out


def decode_step_layers_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                           v_new: torch.Tensor, position_ids: torch.Tensor, out: torch.Tensor | None = None,
                           scale: float | None = None, workspace: torch.Tensor | None = None,
                           max_kv_len_hint: int = 0, err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """decode_step_fwd for every layer of [layers, ...]-stacked inputs and
    caches in one launch (layer l uses q[l], k_cache[l], ..., writes out[l]);
    the layers are independent, a batch of layers * B sequences. A workspace
    must hold decode_attn_workspace_size(layers * B, ...) bytes."""
    if out is None:
        out = torch.empty_like(q)
    _require(q.dim() == 4 and k_cache.dim() == 5, "q must be [layers, B, H, D] and caches [layers, B, Hkv, cap, D]")
    layers = q.shape[0]
    if layers == 0:
        return out
    _require(k_cache.shape[0] == layers and v_cache.shape == k_cache.shape and out.shape == q.shape,
             "every tensor needs the same leading layer count")
    B, H, Hkv, D, cap = _step_inputs(q, k_cache, v_cache, k_new, v_new, position_ids, out, lead=(layers,))
    dev = q.device
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = alloc_workspace(layers * B, H, Hkv, D, cap, dev)
    ws, ws_bytes = _workspace(workspace, dev)
    _call("decode_step_layers_fwd", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
          _ptr(position_ids), layers, B, H, Hkv, D, cap, float(scale), _ptr(out), ws, ws_bytes,
          int(max_kv_len_hint), _dtype_code(q), _err_ptr(err_flag, dev), _stream(q))
    return out


_thread_state = threading.local()  # mirror of the library's per-thread ordering promise


def set_prefix_ready(on: bool) -> None:
    """Ordering promise of this thread's later decode calls (see
    da_set_prefix_ready in the C header): with B == 1 and a length bound, no
    kernel still running when a call's kernel starts writes the cache rows the
    call reads, so the kernel may copy its first tiles before waiting for the
    previous kernel on the stream."""
    load_library().da_set_prefix_ready(1 if on else 0)
    _thread_state.prefix_ready = bool(on)


@contextlib.contextmanager
def prefix_ready():
    """set_prefix_ready(True) for the calls (or the stream capture) inside the
    block; the thread's previous setting comes back on exit (blocks nest)."""
    before = getattr(_thread_state, "prefix_ready", False)
    set_prefix_ready(True)
    try:
        yield
    finally:
        set_prefix_ready(before)


def test_skip_slot(slot: int) -> None:
    """Failure-detection test hook: with slot >= 0, later decode calls of this
    thread leave that ring slot of one CTA unfilled, so its bounded waits
    expire and the call reports DA_DEVERR_TIMEOUT (-1 turns it off)."""
    load_library().da_test_skip_slot(int(slot))


STATIC_SCRATCH_BYTES = 1 << 20  # DA_STATIC_SCRATCH_BYTES of the C header


def decode_attn_fwd_static_scratch(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   kv_len: torch.Tensor, out: torch.Tensor | None = None,
                                   scale: float | None = None, max_kv_len_hint: int = 0,
                                   err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """decode_attn_fwd without a caller workspace: the library's own fixed
    device scratch array holds the split partials (for callers that may not
    allocate GPU memory). ``out`` must be given by such callers; when it is
    None this helper creates it with torch for convenience."""
    if out is None:
        out = torch.empty_like(q)
    B, H, Hkv, D, cap = _attn_shapes(q, k_cache, v_cache, out)
    dev = q.device
    _on(dev, kv_len=kv_len)
    _require(kv_len.dtype == torch.int32 and kv_len.numel() == B, "kv_len must be int32 [B]")
    if scale is None:
        scale = D ** -0.5
    _call("decode_attn_fwd_static_scratch", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), B, H, Hkv, D,
          cap, float(scale), _ptr(out), int(max_kv_len_hint), _dtype_code(q), _err_ptr(err_flag, dev), _stream(q))
    return out
