"""Thin ctypes binding over libfw_attn.so (the C ABI in include/fw_attn.h).

Argument marshalling only: torch tensors become fw_tensor_t views (device
pointer, dtype, shape, strides in elements) and the current torch CUDA stream
is passed through.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback path.  A missing or unbuilt library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfw_attn.so")

FW_OK, FW_ERR_INVALID_ARG, FW_ERR_UNSUPPORTED, FW_ERR_WORKSPACE, FW_ERR_CUDA, FW_ERR_DEVICE_TIMEOUT = range(6)
STATUS_NAMES = {0: "FW_OK", 1: "FW_ERR_INVALID_ARG", 2: "FW_ERR_UNSUPPORTED", 3: "FW_ERR_WORKSPACE",
                4: "FW_ERR_CUDA", 5: "FW_ERR_DEVICE_TIMEOUT"}
FW_BF16, FW_F32, FW_I32, FW_FP8_E4M3 = 0, 1, 2, 3
FW_OPT_DECODE_CHUNK_TOKENS, FW_OPT_WAIT_TIMEOUT_MS, FW_OPT_KERNEL_TIMING, FW_OPT_MAX_CTAS = 0, 1, 2, 3
FW_OPT_PREFILL_SOFTMAX, FW_OPT_TEST_STALL = 4, 5
FW_COUNTER_PREFILL_REPLAYS, FW_COUNTER_LATENT_RESCALES = 0, 1

_DTYPES = {torch.bfloat16: FW_BF16, torch.float32: FW_F32, torch.int32: FW_I32,
           torch.float8_e4m3fn: FW_FP8_E4M3}


class FwError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class FwTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class FwDecodePlan(ctypes.Structure):
    _fields_ = [("group", ctypes.c_int32), ("rows_per_unit", ctypes.c_int32),
                ("tokens_per_unit", ctypes.c_int32), ("heads_per_unit", ctypes.c_int32),
                ("row_groups", ctypes.c_int32), ("min_span_tiles", ctypes.c_int32),
                ("max_pieces", ctypes.c_int32), ("num_units", ctypes.c_int64),
                ("partial_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("grid", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None):
    """Load libfw_attn.so (built in-tree by build.py); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run ragged_softmax_attention_gb300.build.build() "
                           "(nvcc, sm_103a) first -- there is no fallback implementation")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FwTensor)
    S = ctypes.c_int
    lib.fw_paged_decode.restype = S
    lib.fw_paged_decode.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.fw_paged_decode_noalloc.restype = S
    lib.fw_paged_decode_noalloc.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.fw_paged_decode_window.restype = ctypes.c_int
    lib.fw_paged_decode_window.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int32, P, P, ctypes.c_void_p]
    lib.fw_paged_decode_masked.restype = ctypes.c_int
    lib.fw_paged_decode_masked.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_float, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.fw_kv_append.restype = ctypes.c_int
    lib.fw_kv_append.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
    lib.fw_paged_decode_append.restype = ctypes.c_int
    lib.fw_paged_decode_append.argtypes = [P, P, P, P, ctypes.c_int64, P, P, P, P, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_int32, P, P, ctypes.c_void_p]
    lib.fw_paged_decode_fp8.restype = ctypes.c_int
    lib.fw_paged_decode_fp8.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float, P, P,
                                        ctypes.c_void_p]
    lib.fw_paged_decode_workspace_size.restype = S
    lib.fw_paged_decode_workspace_size.argtypes = [P, P, P, P, ctypes.POINTER(ctypes.c_size_t)]
    lib.fw_varlen_prefill.restype = S
    lib.fw_varlen_prefill.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.fw_set_workspace.restype = S
    lib.fw_set_workspace.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.fw_get_device_status.restype = S
    lib.fw_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.fw_last_error.restype = ctypes.c_char_p
    lib.fw_last_error.argtypes = []
    lib.fw_set_option.restype = S
    lib.fw_set_option.argtypes = [ctypes.c_int32, ctypes.c_int64]
    lib.fw_kernel_timing_read.restype = S
    lib.fw_kernel_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    lib.fw_read_counters.restype = S
    lib.fw_read_counters.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]
    lib.fw_launch_count.restype = ctypes.c_int64
    lib.fw_launch_count.argtypes = []
    lib.fw_plan_decode.restype = S
    lib.fw_plan_decode.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_int64, ctypes.c_int32,
                                                          ctypes.POINTER(FwDecodePlan)]
    _lib = lib
    return lib


def _check(status: int):
    if status != FW_OK:
        raise FwError(status, load_library().fw_last_error().decode(errors="replace"))


def as_fw_tensor(t: Optional[torch.Tensor]):
    """fw_tensor_t view of a torch tensor (no copy).  None -> NULL pointer."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 5:
        raise ValueError("at most 5 dimensions")
    ft = FwTensor()
    ft.data = t.data_ptr() if t.numel() > 0 else None
    ft.dtype = _DTYPES[t.dtype]
    ft.ndim = t.dim()
    for i in range(t.dim()):
        ft.shape[i] = t.shape[i]
        ft.stride[i] = t.stride(i)
    return ft


def _ref(ft):
    return ctypes.byref(ft) if ft is not None else None


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale, out=None, lse=None,
                 return_lse=True, stream=None):
    """fw_paged_decode: returns (out [B, q_len, Hq, Dv] bf16, lse [B, q_len, Hq] f32 or None)."""
    lib = load_library()
    B, q_len, Hq, _ = q.shape
    Dv = v_cache.shape[3]
    if out is None:
        out = torch.empty((B, q_len, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode(*[_ref(a) for a in args], ctypes.c_float(scale), _ref(fo), _ref(fl),
                               _stream_handle(stream)))
    return out, lse


def paged_decode_fp8(q, k_cache, v_cache, block_table, seq_lens, scale, k_scale, v_scale, out=None, lse=None,
                     return_lse=True, stream=None):
    """fw_paged_decode_fp8: FP8 E4M3 caches (torch.float8_e4m3fn) with one scale
    each; returns (out [B, q_len, Hq, Dv] bf16, lse [B, q_len, Hq] f32 or None)."""
    lib = load_library()
    B, q_len, Hq, _ = q.shape
    Dv = v_cache.shape[3]
    if out is None:
        out = torch.empty((B, q_len, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode_fp8(*[_ref(a) for a in args], ctypes.c_float(scale), ctypes.c_float(k_scale),
                                   ctypes.c_float(v_scale), _ref(fo), _ref(fl), _stream_handle(stream)))
    return out, lse


def paged_decode_window(q, k_cache, v_cache, block_table, seq_lens, scale, window_left, k_scale=1.0, v_scale=1.0,
                        out=None, lse=None, return_lse=True, stream=None):
    """fw_paged_decode_window: token t of row b sees keys max(0, n - q_len + t -
    window_left) .. n - q_len + t (window_left = -1: no window); BF16 or FP8
    E4M3 caches (the scales apply to FP8 caches and must be 1 for BF16).
    Returns (out [B, q_len, Hq, Dv] bf16, lse [B, q_len, Hq] f32 or None)."""
    lib = load_library()
    B, q_len, Hq, _ = q.shape
    Dv = v_cache.shape[3]
    if out is None:
        out = torch.empty((B, q_len, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode_window(*[_ref(a) for a in args], ctypes.c_float(scale), ctypes.c_float(k_scale),
                                      ctypes.c_float(v_scale), ctypes.c_int32(window_left), _ref(fo), _ref(fl),
                                      _stream_handle(stream)))
    return out, lse


def paged_decode_masked(q, k_cache, v_cache, block_table, seq_lens, scale, causal=True, window_left=-1, k_scale=1.0,
                        v_scale=1.0, out=None, lse=None, return_lse=True, stream=None):
    """fw_paged_decode_masked: causal=True, token t of row b sees keys up to
    n - q_len + t; causal=False, all n keys; a window_left >= 0 starts either
    range at max(0, n - q_len + t - window_left).  BF16 or FP8 E4M3 caches.
    Returns (out [B, q_len, Hq, Dv] bf16, lse [B, q_len, Hq] f32 or None)."""
    lib = load_library()
    B, q_len, Hq, _ = q.shape
    Dv = v_cache.shape[3]
    if out is None:
        out = torch.empty((B, q_len, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode_masked(*[_ref(a) for a in args], ctypes.c_float(scale), ctypes.c_int32(1 if causal else 0),
                                      ctypes.c_int32(window_left), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
                                      _ref(fo), _ref(fl), _stream_handle(stream)))
    return out, lse


def kv_append(k_new, v_new, slot_mapping, layer_base_rows, k_cache, v_cache, k_scale=1.0, v_scale=1.0, stream=None):
    """fw_kv_append: token (b, t) of k_new / v_new [B, q_len, Hkv, D] (bf16) goes
    to cache token row layer_base_rows + max(slot_mapping[b * q_len + t], 0) of
    k_cache / v_cache [pages, ps, Hkv, D] (bf16, or float8_e4m3fn storing
    E4M3(x / scale)); the caches are written in place.  v_new and v_cache may
    both be None."""
    lib = load_library()
    t = [as_fw_tensor(x) if x is not None else None for x in (k_new, v_new, slot_mapping, k_cache, v_cache)]
    _check(lib.fw_kv_append(_ref(t[0]), _ref(t[1]), _ref(t[2]), ctypes.c_int64(layer_base_rows), _ref(t[3]),
                            _ref(t[4]), ctypes.c_float(k_scale), ctypes.c_float(v_scale), _stream_handle(stream)))


def paged_decode_append(q, k_new, v_new, slot_mapping, layer_base_rows, k_cache, v_cache, block_table, seq_lens,
                        scale, k_scale=1.0, v_scale=1.0, window_left=-1, out=None, lse=None, return_lse=True,
                        stream=None):
    """fw_paged_decode_append: kv_append into the (packed) caches, then the
    decode of the layer whose pages start at layer_base_rows / ps (block_table
    counts from there).  Returns (out, lse)."""
    lib = load_library()
    B, q_len, Hq, _ = q.shape
    Dv = v_cache.shape[3]
    if out is None:
        out = torch.empty((B, q_len, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    t = [as_fw_tensor(x) for x in (q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode_append(_ref(t[0]), _ref(t[1]), _ref(t[2]), _ref(t[3]), ctypes.c_int64(layer_base_rows),
                                      _ref(t[4]), _ref(t[5]), _ref(t[6]), _ref(t[7]), ctypes.c_float(scale),
                                      ctypes.c_float(k_scale), ctypes.c_float(v_scale), ctypes.c_int32(window_left),
                                      _ref(fo), _ref(fl), _stream_handle(stream)))
    return out, lse


def paged_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse=None, stream=None):
    """fw_paged_decode_noalloc: the same decode without any device allocation.

    For callers that may not allocate device memory (a runtime that owns the
    whole pool, a loop that cannot afford cudaMalloc's synchronisation): the
    output buffers are the caller's, and the scratch is the library's fixed
    64 MiB device array.  Calls overlapping on the GPU race on that array.
    """
    lib = load_library()
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table, seq_lens)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_paged_decode_noalloc(*[_ref(a) for a in args], ctypes.c_float(scale), _ref(fo), _ref(fl),
                                       _stream_handle(stream)))
    return out, lse


def paged_decode_workspace_size(q, k_cache, v_cache, block_table) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    args = [as_fw_tensor(x) for x in (q, k_cache, v_cache, block_table)]
    _check(lib.fw_paged_decode_workspace_size(*[_ref(a) for a in args], ctypes.byref(n)))
    return n.value


def varlen_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, causal, scale, out=None, lse=None,
                   return_lse=True, stream=None):
    """fw_varlen_prefill: returns (out [total_q, Hq, Dv] bf16, lse [total_q, Hq] f32 or None)."""
    lib = load_library()
    total_q, Hq, _ = q.shape
    Dv = v.shape[2]
    if out is None:
        out = torch.empty((total_q, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    args = [as_fw_tensor(x) for x in (q, k, v, cu_seqlens_q, cu_seqlens_k)]
    fo, fl = as_fw_tensor(out), as_fw_tensor(lse)
    _check(lib.fw_varlen_prefill(*[_ref(a) for a in args], int(bool(causal)), ctypes.c_float(scale),
                                 _ref(fo), _ref(fl), _stream_handle(stream)))
    return out, lse


def set_workspace(buf: Optional[torch.Tensor], stream=None):
    lib = load_library()
    if buf is None:
        _check(lib.fw_set_workspace(None, 0, None))
    else:
        _check(lib.fw_set_workspace(buf.data_ptr(), buf.numel() * buf.element_size(), _stream_handle(stream)))


def device_status(stream=None) -> int:
    lib = load_library()
    code = ctypes.c_int32(0)
    _check(lib.fw_get_device_status(_stream_handle(stream), ctypes.byref(code)))
    return code.value


def set_option(option: int, value: int):
    _check(load_library().fw_set_option(option, int(value)))


def kernel_timing_read():
    lib = load_library()
    ms = ctypes.c_double(0)
    n = ctypes.c_int64(0)
    _check(lib.fw_kernel_timing_read(ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def read_counters(stream=None) -> dict:
    """Device event counters since the last read (which resets them):
    {"prefill_replays": ..., "latent_rescales": ...}."""
    vals = (ctypes.c_int64 * 2)()
    _check(load_library().fw_read_counters(_stream_handle(stream), vals, 2))
    return {"prefill_replays": vals[FW_COUNTER_PREFILL_REPLAYS], "latent_rescales": vals[FW_COUNTER_LATENT_RESCALES]}


def launch_count() -> int:
    return int(load_library().fw_launch_count())


def plan_decode(batch, q_len, num_q_heads, num_kv_heads, head_dim_v, max_kv_len, num_sms=0) -> dict:
    plan = FwDecodePlan()
    _check(load_library().fw_plan_decode(batch, q_len, num_q_heads, num_kv_heads, head_dim_v,
                                         max_kv_len, num_sms, ctypes.byref(plan)))
    return {name: getattr(plan, name) for name, _ in FwDecodePlan._fields_}
