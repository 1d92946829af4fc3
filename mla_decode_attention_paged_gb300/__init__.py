"""Paged MLA decode attention for one GB300 (sm_103a): the Python binding of
libmla_gb300, whose C ABI is declared in include/mla.h.

The binding only marshals arguments: it checks tensor dtypes, shapes and
devices, passes raw pointers and the current CUDA stream to the library, and
turns status codes into exceptions.  Every step of the computation runs in
the library's CUDA kernels.  There is no fallback: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "MLAError", "Dims", "dims", "load_library", "check_dims", "cache_append", "auto_num_splits",
    "decode_workspace_size", "decode", "decode_multi_workspace_size", "decode_multi", "decode_sparse_workspace_size",
    "decode_sparse", "decode_no_alloc", "combine", "read_device_status", "read_status_word",
    "set_timing_events", "status_string", "version",
    "MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_WORKSPACE", "MLA_ERR_CUDA",
    "MLA_ERR_DEVICE_TIMEOUT", "MLA_ERR_DEVICE_BOUNDS", "MLA_CACHE_BF16", "MLA_CACHE_INT8", "MLA_CACHE_FP8",
    "MAX_Q_LEN", "MAX_TOP_K", "MAX_PREFILL_CHUNK",
]

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_CUDA = -4
MLA_ERR_DEVICE_TIMEOUT = -5
MLA_ERR_DEVICE_BOUNDS = -6
MLA_CACHE_BF16 = 0
MLA_CACHE_INT8 = 1
MLA_CACHE_FP8 = 2
MAX_Q_LEN = 8  # MLA_MAX_Q_LEN in include/mla.h
MAX_PREFILL_CHUNK = 2048  # MLA_MAX_PREFILL_CHUNK in include/mla.h
MAX_TOP_K = 1 << 20  # MLA_MAX_TOP_K in include/mla.h

# every function include/mla.h declares
EXPORTED_SYMBOLS = (
    "mla_check_dims", "mla_cache_append", "mla_auto_num_splits", "mla_decode_workspace_size",
    "mla_decode", "mla_combine", "mla_read_device_status", "mla_read_status_word",
    "mla_status_string", "mla_set_timing_events", "mla_version", "mla_decode_no_alloc",
    "mla_test_inject_wait_timeout", "mla_decode_multi_workspace_size", "mla_decode_multi",
    "mla_decode_sparse_workspace_size", "mla_decode_sparse", "mla_test_force_single_cta",
    "mla_prefill_workspace_size", "mla_prefill",
)
NO_ALLOC_WORKSPACE_BYTES = 16 << 20  # MLA_NO_ALLOC_WORKSPACE_BYTES in include/mla.h


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("qk_nope_dim", ctypes.c_int32),
                ("v_head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32)]


def dims(num_heads: int, page_size: int, int8: bool = False, kv_lora_rank: int = 512, rope_dim: int = 64,
         qk_nope_dim: int = 128, v_head_dim: int = 128, fp8: bool = False) -> Dims:
    """Model dimensions; ``int8`` / ``fp8`` select a 1-byte cache (INT8 codes, or
    FP8 E4M3 codes held as uint8 or torch.float8_e4m3fn) with per-token scales."""
    if int8 and fp8:
        raise ValueError("int8 and fp8 are exclusive")
    code = MLA_CACHE_INT8 if int8 else MLA_CACHE_FP8 if fp8 else MLA_CACHE_BF16
    return Dims(num_heads, kv_lora_rank, rope_dim, qk_nope_dim, v_head_dim, page_size, code)


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32


def load_library(build_if_missing: bool = False, path: str | None = None):
    """Load libmla_gb300.so (building it first if asked and it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mla_decode_attention_paged_gb300.build`")
    lib = ctypes.CDLL(path)
    DP = ctypes.POINTER(Dims)
    sig = {
        "mla_check_dims": (_I, [DP]),
        "mla_cache_append": (_I, [DP, _P, _P, _I, _P, _I, _I, _P, _P, _I, _P, _P, ctypes.c_double, _P, _P]),
        "mla_auto_num_splits": (_I, [DP, _I]),
        "mla_decode_workspace_size": (ctypes.c_size_t, [DP, _I, _I]),
        "mla_decode": (_I, [DP, _P, _P, _P, _P, _I, _P, _I, _P, _I, _P, _P, ctypes.c_float, _I, _P,
                            ctypes.c_size_t, _P, _P, _P]),
        "mla_decode_multi_workspace_size": (ctypes.c_size_t, [DP, _I, _I, _I]),
        "mla_decode_multi": (_I, [DP, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_float, _I, _P,
                                  ctypes.c_size_t, _P, _P, _P]),
        "mla_decode_sparse_workspace_size": (ctypes.c_size_t, [DP, _I, _I, _I]),
        "mla_decode_sparse": (_I, [DP, _P, _P, _P, _P, _I, _P, _I, _P, _I, _P, _I, _P, _P, ctypes.c_float, _I, _P,
                                   ctypes.c_size_t, _P, _P, _P]),
        "mla_decode_no_alloc": (_I, [DP, _P, _P, _P, _P, _I, _P, _I, _P, _I, _P, _P, ctypes.c_float, _I, _P, _P,
                                     _P, _P]),
        "mla_combine": (_I, [DP, _P, _P, _I, _I, _P, _P, _P]),
        "mla_read_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
        "mla_read_status_word": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
        "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mla_set_timing_events": (_I, [_P, _P]),
        "mla_version": (ctypes.c_int, []),
        "mla_test_inject_wait_timeout": (_I, [_I]),
        "mla_test_force_single_cta": (_I, [_I]),
        "mla_prefill_workspace_size": (ctypes.c_size_t, [DP, _I, _I, _I]),
        "mla_prefill": (_I, [DP, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_double, _P, _P, _P, _P,
                             ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _L():
    return _lib if _lib is not None else load_library()


def status_string(status: int) -> str:
    return _L().mla_status_string(int(status)).decode()


def version() -> int:
    return _L().mla_version()


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MLAError(status, what)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor", device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _cache_ptrs(d: Dims, cache: torch.Tensor, scale_zero: torch.Tensor | None, device=None):
    """Pointers of the cache rows (bf16 values, int8 codes, or E4M3 codes) and of
    their per-token scales (None for bf16 caches)."""
    if d.cache_dtype == MLA_CACHE_FP8:
        if isinstance(cache, torch.Tensor) and cache.dtype == torch.float8_e4m3fn:
            cache = cache.view(torch.uint8)
        want = torch.uint8
    else:
        want = torch.int8 if d.cache_dtype == MLA_CACHE_INT8 else torch.bfloat16
    byte = d.cache_dtype != MLA_CACHE_BF16
    return (_ptr(cache, want, "cache", device),
            _ptr(scale_zero, torch.float32, "scale_zero", device) if byte else None)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def check_dims(d: Dims) -> int:
    return _L().mla_check_dims(ctypes.byref(d))


def cache_append(d: Dims, cache: torch.Tensor, scale_zero: torch.Tensor | None, block_table: torch.Tensor,
                 seq_ids: torch.Tensor, positions: torch.Tensor, c_kv: torch.Tensor, k_pe: torch.Tensor,
                 rope_theta: float = 10000.0, device_status: torch.Tensor | None = None, stream=None) -> None:
    """mla_cache_append: write new tokens' rows into the paged cache (in place)."""
    dev = cache.device
    st = _L().mla_cache_append(
        ctypes.byref(d), *_cache_ptrs(d, cache, scale_zero, dev), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table", dev), block_table.shape[0], block_table.shape[1],
        _ptr(seq_ids, torch.int32, "seq_ids", dev), _ptr(positions, torch.int32, "positions", dev),
        seq_ids.numel(), _ptr(c_kv, torch.bfloat16, "c_kv", dev), _ptr(k_pe, torch.bfloat16, "k_pe", dev),
        float(rope_theta), _ptr(device_status, torch.int32, "device_status", dev), _stream(stream))
    _check(st, "mla_cache_append")


def auto_num_splits(d: Dims, batch: int) -> int:
    n = _L().mla_auto_num_splits(ctypes.byref(d), int(batch))
    if n < 0:
        raise MLAError(n, "mla_auto_num_splits")
    return n


def decode_workspace_size(d: Dims, batch: int, num_splits: int = 0) -> int:
    n = _L().mla_decode_workspace_size(ctypes.byref(d), int(batch), int(num_splits))
    if n == 0:
        raise MLAError(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size")
    return n


def decode(d: Dims, q_nope, q_pe, cache, scale_zero, block_table, seq_lens, W_UK, W_UV, softmax_scale: float,
           num_splits: int = 0, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
           lse_out: torch.Tensor | None = None, want_lse: bool = True, stream=None):
    """mla_decode: one decode step; returns (out bf16 [B, H, 128], lse fp32 [B, H] or None).

    If ``workspace`` is None a uint8 buffer of the required size is taken from
    torch's allocator here (the library itself never allocates)."""
    B = q_nope.shape[0]
    dev = q_nope.device
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(d, B, num_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((B, d.num_heads, d.v_head_dim), dtype=torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, d.num_heads), dtype=torch.float32, device=dev)
    st = _L().mla_decode(
        ctypes.byref(d), _ptr(q_nope, torch.bfloat16, "q_nope"), _ptr(q_pe, torch.bfloat16, "q_pe", dev),
        *_cache_ptrs(d, cache, scale_zero, dev), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table", dev), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens", dev), B, _ptr(W_UK, torch.bfloat16, "W_UK", dev),
        _ptr(W_UV, torch.bfloat16, "W_UV", dev), float(softmax_scale), int(num_splits),
        _ptr(workspace, None, "workspace", dev), workspace.numel() * workspace.element_size(),
        _ptr(out, torch.bfloat16, "out", dev), _ptr(lse_out, torch.float32, "lse_out", dev), _stream(stream))
    _check(st, "mla_decode")
    return out, lse_out


def decode_multi_workspace_size(d: Dims, batch: int, q_len: int, num_splits: int = 0) -> int:
    n = _L().mla_decode_multi_workspace_size(ctypes.byref(d), int(batch), int(q_len), int(num_splits))
    if n == 0:
        raise MLAError(MLA_ERR_INVALID_ARG, "mla_decode_multi_workspace_size")
    return n


def decode_multi(d: Dims, q_nope, q_pe, cache, scale_zero, block_table, seq_lens, W_UK, W_UV,
                 softmax_scale: float, num_splits: int = 0, workspace: torch.Tensor | None = None,
                 out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None, want_lse: bool = True,
                 stream=None):
    """mla_decode_multi: q_len = q_nope.shape[1] query tokens per sequence (the
    last q_len tokens of each cache, causal among themselves); q_nope bf16
    [B, T, H, 128], q_pe bf16 [B, T, H, 64].  Returns (out bf16 [B, T, H, 128],
    lse fp32 [B, T, H] or None)."""
    B, T = q_nope.shape[0], q_nope.shape[1]
    dev = q_nope.device
    if workspace is None:
        workspace = torch.empty(decode_multi_workspace_size(d, B, T, num_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((B, T, d.num_heads, d.v_head_dim), dtype=torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, T, d.num_heads), dtype=torch.float32, device=dev)
    st = _L().mla_decode_multi(
        ctypes.byref(d), _ptr(q_nope, torch.bfloat16, "q_nope"), _ptr(q_pe, torch.bfloat16, "q_pe", dev),
        *_cache_ptrs(d, cache, scale_zero, dev), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table", dev), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens", dev), B, T, _ptr(W_UK, torch.bfloat16, "W_UK", dev),
        _ptr(W_UV, torch.bfloat16, "W_UV", dev), float(softmax_scale), int(num_splits),
        _ptr(workspace, None, "workspace", dev), workspace.numel() * workspace.element_size(),
        _ptr(out, torch.bfloat16, "out", dev), _ptr(lse_out, torch.float32, "lse_out", dev), _stream(stream))
    _check(st, "mla_decode_multi")
    return out, lse_out


def prefill_workspace_size(d: Dims, batch: int, chunk: int, num_splits: int = 0) -> int:
    n = _L().mla_prefill_workspace_size(ctypes.byref(d), int(batch), int(chunk), int(num_splits))
    if n == 0:
        raise MLAError(MLA_ERR_INVALID_ARG, "mla_prefill_workspace_size")
    return n


def prefill(d: Dims, cache, scale_zero, block_table, seq_lens, c_kv, k_pe, q_nope, q_pe, W_UK, W_UV,
            softmax_scale: float, rope_theta: float = 10000.0, num_splits: int = 0,
            workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
            lse_out: torch.Tensor | None = None, want_lse: bool = True, stream=None):
    """mla_prefill: one chunk of chunk = q_nope.shape[1] tokens per sequence,
    at positions seq_lens[b] - chunk .. seq_lens[b] - 1.  Writes c_kv bf16
    [B, chunk, 512] / k_pe bf16 [B, chunk, 64] into the cache, then attends
    q_nope bf16 [B, chunk, H, 128] / q_pe [B, chunk, H, 64] causally.  Returns
    (out bf16 [B, chunk, H, 128], lse fp32 [B, chunk, H] or None)."""
    B, T = q_nope.shape[0], q_nope.shape[1]
    dev = q_nope.device
    if workspace is None:
        workspace = torch.empty(prefill_workspace_size(d, B, T, num_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((B, T, d.num_heads, d.v_head_dim), dtype=torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, T, d.num_heads), dtype=torch.float32, device=dev)
    cache_p, scale_p = _cache_ptrs(d, cache, scale_zero, dev)
    st = _L().mla_prefill(
        ctypes.byref(d), cache_p, scale_p, cache.shape[0], _ptr(block_table, torch.int32, "block_table", dev),
        block_table.shape[1], _ptr(seq_lens, torch.int32, "seq_lens", dev), B, T,
        _ptr(c_kv, torch.bfloat16, "c_kv", dev), _ptr(k_pe, torch.bfloat16, "k_pe", dev), float(rope_theta),
        _ptr(q_nope, torch.bfloat16, "q_nope", dev), _ptr(q_pe, torch.bfloat16, "q_pe", dev),
        _ptr(W_UK, torch.bfloat16, "W_UK", dev), _ptr(W_UV, torch.bfloat16, "W_UV", dev), float(softmax_scale),
        int(num_splits), _ptr(workspace, None, "workspace", dev), workspace.numel() * workspace.element_size(),
        _ptr(out, torch.bfloat16, "out", dev), _ptr(lse_out, torch.float32, "lse_out", dev), _stream(stream))
    _check(st, "mla_prefill")
    return out, lse_out


def decode_sparse_workspace_size(d: Dims, batch: int, top_k: int, num_splits: int = 0) -> int:
    n = _L().mla_decode_sparse_workspace_size(ctypes.byref(d), int(batch), int(top_k), int(num_splits))
    if n == 0:
        raise MLAError(MLA_ERR_INVALID_ARG, "mla_decode_sparse_workspace_size")
    return n


def decode_sparse(d: Dims, q_nope, q_pe, cache, scale_zero, block_table, seq_lens, token_indices, W_UK, W_UV,
                  softmax_scale: float, num_splits: int = 0, workspace: torch.Tensor | None = None,
                  out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None, want_lse: bool = True,
                  stream=None):
    """mla_decode_sparse: attention over the listed positions of each sequence
    (token_indices int32 [B, top_k], -1 = padding).  Returns (out bf16
    [B, H, 128], lse fp32 [B, H] or None)."""
    B, K = token_indices.shape
    dev = q_nope.device
    if workspace is None:
        workspace = torch.empty(decode_sparse_workspace_size(d, B, K, num_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((B, d.num_heads, d.v_head_dim), dtype=torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, d.num_heads), dtype=torch.float32, device=dev)
    st = _L().mla_decode_sparse(
        ctypes.byref(d), _ptr(q_nope, torch.bfloat16, "q_nope"), _ptr(q_pe, torch.bfloat16, "q_pe", dev),
        *_cache_ptrs(d, cache, scale_zero, dev), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table", dev), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens", dev), B, _ptr(token_indices, torch.int32, "token_indices", dev), K,
        _ptr(W_UK, torch.bfloat16, "W_UK", dev), _ptr(W_UV, torch.bfloat16, "W_UV", dev), float(softmax_scale),
        int(num_splits), _ptr(workspace, None, "workspace", dev), workspace.numel() * workspace.element_size(),
        _ptr(out, torch.bfloat16, "out", dev), _ptr(lse_out, torch.float32, "lse_out", dev), _stream(stream))
    _check(st, "mla_decode_sparse")
    return out, lse_out


def decode_no_alloc(d: Dims, q_nope, q_pe, cache, scale_zero, block_table, seq_lens, W_UK, W_UV,
                    softmax_scale: float, num_splits: int = 0, out: torch.Tensor | None = None,
                    lse_out: torch.Tensor | None = None, device_status: torch.Tensor | None = None, stream=None):
    """mla_decode_no_alloc: mla_decode on the library's fixed scratch array, for
    callers that cannot allocate device memory (outputs are still the
    caller's).  Returns (out, lse)."""
    B = q_nope.shape[0]
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, d.num_heads, d.v_head_dim), dtype=torch.bfloat16, device=dev)
    st = _L().mla_decode_no_alloc(
        ctypes.byref(d), _ptr(q_nope, torch.bfloat16, "q_nope"), _ptr(q_pe, torch.bfloat16, "q_pe", dev),
        *_cache_ptrs(d, cache, scale_zero, dev), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table", dev), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens", dev), B, _ptr(W_UK, torch.bfloat16, "W_UK", dev),
        _ptr(W_UV, torch.bfloat16, "W_UV", dev), float(softmax_scale), int(num_splits),
        _ptr(out, torch.bfloat16, "out", dev), _ptr(lse_out, torch.float32, "lse_out", dev),
        _ptr(device_status, torch.int32, "device_status", dev), _stream(stream))
    _check(st, "mla_decode_no_alloc")
    return out, lse_out


def combine(d: Dims, partial_o: torch.Tensor, partial_lse: torch.Tensor, o_lat_out=None, lse_out=None,
            stream=None):
    """mla_combine over [B, S, H, 512] partials; returns (o_lat [B, H, 512], lse [B, H])."""
    B, S, H, D = partial_o.shape
    dev = partial_o.device
    if o_lat_out is None:
        o_lat_out = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, H), dtype=torch.float32, device=dev)
    st = _L().mla_combine(ctypes.byref(d), _ptr(partial_o, torch.float32, "partial_o"),
                          _ptr(partial_lse, torch.float32, "partial_lse", dev), B, S,
                          _ptr(o_lat_out, torch.float32, "o_lat_out", dev), _ptr(lse_out, torch.float32, "lse_out", dev),
                          _stream(stream))
    _check(st, "mla_combine")
    return o_lat_out, lse_out


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(_L().mla_read_device_status(_ptr(workspace, None, "workspace"), ctypes.byref(v), _stream(stream)),
           "mla_read_device_status")
    return v.value


def read_status_word(word: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(_L().mla_read_status_word(_ptr(word, torch.int32, "status word"), ctypes.byref(v), _stream(stream)),
           "mla_read_status_word")
    return v.value


def test_inject_wait_timeout(enable: bool) -> None:
    """Test hook: make the attention kernel's first page wait of each CTA unsatisfiable
    (it times out and the status word reports MLA_ERR_DEVICE_TIMEOUT)."""
    _check(_L().mla_test_inject_wait_timeout(1 if enable else 0), "mla_test_inject_wait_timeout")


def test_force_single_cta(enable: bool) -> None:
    """Test hook: run bf16 decodes on the single-CTA attention kernel (the
    fallback for devices that cannot place CTA pairs)."""
    _check(_L().mla_test_force_single_cta(1 if enable else 0), "mla_test_force_single_cta")


def set_timing_events(start: torch.cuda.Event | None, stop: torch.cuda.Event | None) -> None:
    """Have mla_decode record these events around its attention kernel (None clears)."""
    a = start.cuda_event if start is not None else None
    b = stop.cuda_event if stop is not None else None
    _check(_L().mla_set_timing_events(a, b), "mla_set_timing_events")
