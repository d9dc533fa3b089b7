"""fp64 CPU oracle for ragged softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no
code with it.

Two parts:
  * ``paged_decode`` / ``varlen_prefill``: the plain definition of softmax
    attention over a paged or packed KV store, computed in fp64 by ``oracle.c``
    (see the header there for the passages each step follows);
  * ``planning``: the pages' bookkeeping formulas (task mapping, page/stack
    counts, query folding, packed-query tiles, split-KV workspace size, the
    static-anchor budget), restated independently of the library's planner.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain C, no vector intrinsics)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        D = ctypes.c_double
        lib.oracle_paged_decode.restype = I
        lib.oracle_paged_decode.argtypes = [P, P, P, P, P, P, P, L, P, I, I, I, I, I, I, I, I, I, D,
                                            P, L, P, P, P, I]
        lib.oracle_paged_decode_kv8.restype = I
        lib.oracle_paged_decode_kv8.argtypes = [P, P, P, P, P, P, D, D, P, L, P, I, I, I, I, I, I, I, I, I, D,
                                                P, L, P, P, P, I]
        lib.oracle_paged_decode_window.restype = I
        lib.oracle_paged_decode_window.argtypes = [P, P, P, P, P, P, I, D, D, I, P, L, P, I, I, I, I, I, I, I, I, I,
                                                   D, P, L, P, P, P, I]
        lib.oracle_paged_decode_masked.restype = I
        lib.oracle_paged_decode_masked.argtypes = [P, P, P, P, P, P, I, D, D, I, I, P, L, P, I, I, I, I, I, I, I,
                                                   I, I, D, P, L, P, P, P, I]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_kv_append.restype = I
        lib.oracle_kv_append.argtypes = [P, P, P, P, P, L, P, P, P, P, I, ctypes.c_float, ctypes.c_float,
                                         I, I, I, I, I, I, L]
        lib.oracle_e4m3_to_double.restype = D
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_varlen_prefill.restype = I
        lib.oracle_varlen_prefill.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, D,
                                              P, L, P, P, P, I]
        _lib = lib
    return _lib


def _bf16(t: torch.Tensor) -> torch.Tensor:
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    if t.dtype != torch.bfloat16:
        raise TypeError(f"oracle expects bfloat16 inputs, got {t.dtype}")
    return t


def _strides(t: torch.Tensor) -> np.ndarray:
    return np.ascontiguousarray(np.array(t.stride(), dtype=np.int64))


def _i32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def e4m3_to_double(byte: int) -> float:
    """The oracle's decoding of one OCP FP8 E4M3 byte (NaN for S.1111.111)."""
    return _load().oracle_e4m3_to_double(int(byte) & 0xFF)


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale, rows=None, threads=None,
                 k_scale=1.0, v_scale=1.0, window_left=-1, causal=True, with_absv=False):
    """Softmax attention of every (b, t, h) query row over its paged keys.

    q [B, q_len, Hq, Dk], k_cache [P, ps, Hkv, Dk], v_cache [P, ps, Hkv, Dv]
    (bfloat16, any strides; or float8_e4m3fn caches, whose values are taken
    as k_scale * e4m3 and v_scale * e4m3), block_table [B, max_pages] int32,
    seq_lens [B].  rows: optional flat row ids (b * q_len + t) * Hq + h to
    compute; default all.  window_left >= 0: sliding window, token t sees keys
    max(0, n - q_len + t - window_left) .. n - q_len + t ("TokenSpeed-MLA
    2.0.1", window_left); block-table entries of keys before it are not read.
    causal=False: every token sees all n keys (TokenSpeed's non-causal
    decode), a window still starting at max(0, n - q_len + t - window_left).
    Returns (out [n_rows, Dv] float64, lse [n_rows] float64, natural log);
    with_absv=True adds absv [n_rows, Dv], the softmax-weighted mean of |v|
    per output column (the scale of a kernel's rounding error, see oracle.c).
    """
    lib = _load()
    kv8 = k_cache.dtype == torch.float8_e4m3fn
    if kv8:
        if v_cache.dtype != torch.float8_e4m3fn:
            raise TypeError("FP8 keys need FP8 values")
        q = _bf16(q)
        k_cache = k_cache.detach().cpu().view(torch.uint8)
        v_cache = v_cache.detach().cpu().view(torch.uint8)
    else:
        q, k_cache, v_cache = _bf16(q), _bf16(k_cache), _bf16(v_cache)
    B, q_len, Hq, Dk = q.shape
    P, ps, Hkv, Dk2 = k_cache.shape
    Dv = v_cache.shape[3]
    assert Dk2 == Dk and tuple(v_cache.shape[:3]) == (P, ps, Hkv)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    assert bt.ndim == 2 and bt.shape[0] == B and sl.shape == (B,)
    if rows is None:
        rows_arr = np.arange(B * q_len * Hq, dtype=np.int64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows_arr.size
    out = np.zeros((n, Dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    absv = np.zeros((n, Dv), dtype=np.float64) if with_absv else None
    ap = absv.ctypes.data if with_absv else None
    qs, ks, vs = _strides(q), _strides(k_cache), _strides(v_cache)
    if not causal:
        rc = lib.oracle_paged_decode_masked(
            q.data_ptr(), qs.ctypes.data, k_cache.data_ptr(), ks.ctypes.data,
            v_cache.data_ptr(), vs.ctypes.data, int(kv8), float(k_scale), float(v_scale), 0,
            int(window_left if window_left is not None else -1),
            bt.ctypes.data, bt.shape[1], sl.ctypes.data,
            B, q_len, Hq, Hkv, Dk, Dv, ps, P, bt.shape[1], float(scale),
            rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data, ap,
            int(threads or default_threads()))
    elif window_left is not None and int(window_left) >= 0:
        rc = lib.oracle_paged_decode_window(
            q.data_ptr(), qs.ctypes.data, k_cache.data_ptr(), ks.ctypes.data,
            v_cache.data_ptr(), vs.ctypes.data, int(kv8), float(k_scale), float(v_scale), int(window_left),
            bt.ctypes.data, bt.shape[1], sl.ctypes.data,
            B, q_len, Hq, Hkv, Dk, Dv, ps, P, bt.shape[1], float(scale),
            rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data, ap,
            int(threads or default_threads()))
    elif kv8:
        rc = lib.oracle_paged_decode_kv8(
            q.data_ptr(), qs.ctypes.data, k_cache.data_ptr(), ks.ctypes.data,
            v_cache.data_ptr(), vs.ctypes.data, float(k_scale), float(v_scale),
            bt.ctypes.data, bt.shape[1], sl.ctypes.data,
            B, q_len, Hq, Hkv, Dk, Dv, ps, P, bt.shape[1], float(scale),
            rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data, ap,
            int(threads or default_threads()))
    else:
        rc = lib.oracle_paged_decode(
            q.data_ptr(), qs.ctypes.data, k_cache.data_ptr(), ks.ctypes.data,
            v_cache.data_ptr(), vs.ctypes.data, bt.ctypes.data, bt.shape[1], sl.ctypes.data,
            B, q_len, Hq, Hkv, Dk, Dv, ps, P, bt.shape[1], float(scale),
            rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data, ap,
            int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode failed with code {rc}")
    return (out, lse, absv) if with_absv else (out, lse)


def e4m3_from_float(x: float) -> int:
    """The oracle's E4M3 code of an FP32 value: nearest, ties to even,
    saturating to +-448, NaN to S.1111.111."""
    return int(_load().oracle_e4m3_from_float(float(x)))


def kv_append(k_new, v_new, slot_mapping, layer_base_rows, k_cache, v_cache, k_scale=1.0, v_scale=1.0):
    """KV-cache append ("Writing Page Attention with PyPTO", section 4.3): row
    (b, t) of k_new / v_new [B, q_len, Hkv, D] (bfloat16) goes to token row
    layer_base_rows + max(slot_mapping[b * q_len + t], 0) of the caches
    [pages, ps, Hkv, D] (bfloat16, or float8_e4m3fn taking x / scale).
    Returns updated copies (k_cache, v_cache); the inputs are not modified."""
    lib = _load()
    k_new, v_new = _bf16(k_new), _bf16(v_new)
    kv8 = k_cache.dtype == torch.float8_e4m3fn
    kc = k_cache.detach().cpu().clone()
    vc = v_cache.detach().cpu().clone()
    if kv8:
        kc_raw, vc_raw = kc.view(torch.uint8), vc.view(torch.uint8)
    else:
        kc_raw, vc_raw = _bf16(kc), _bf16(vc)
    B, q_len, Hkv, Dk = k_new.shape
    Dv = v_new.shape[3]
    P, ps = kc.shape[0], kc.shape[1]
    sm = _i32(slot_mapping).reshape(-1)
    assert sm.size == B * q_len
    kns, vns, ks, vs = _strides(k_new), _strides(v_new), _strides(kc_raw), _strides(vc_raw)
    rc = lib.oracle_kv_append(k_new.data_ptr(), kns.ctypes.data, v_new.data_ptr(), vns.ctypes.data,
                              sm.ctypes.data, int(layer_base_rows), kc_raw.data_ptr(), ks.ctypes.data,
                              vc_raw.data_ptr(), vs.ctypes.data, int(kv8), float(k_scale), float(v_scale),
                              B, q_len, Hkv, Dk, Dv, ps, P)
    if rc != 0:
        raise ValueError(f"oracle_kv_append failed with code {rc}")
    return kc, vc


def varlen_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, causal, scale, rows=None, threads=None, with_absv=False):
    """Softmax attention of every packed query row over its own sequence's keys.

    q [total_q, Hq, Dk], k [total_k, Hkv, Dk], v [total_k, Hkv, Dv] bfloat16;
    cu_seqlens_q / cu_seqlens_k [B+1].  rows: optional flat ids token * Hq + h.
    Returns (out [n_rows, Dv] float64, lse [n_rows] float64, natural log);
    with_absv=True adds absv [n_rows, Dv] as in paged_decode.
    """
    lib = _load()
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    total_q, Hq, Dk = q.shape
    total_k, Hkv, Dk2 = k.shape
    Dv = v.shape[2]
    assert Dk2 == Dk and tuple(v.shape[:2]) == (total_k, Hkv)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    B = cq.size - 1
    assert ck.size == B + 1 and cq[-1] == total_q and ck[-1] <= total_k
    if rows is None:
        rows_arr = np.arange(total_q * Hq, dtype=np.int64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows_arr.size
    out = np.zeros((n, Dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    absv = np.zeros((n, Dv), dtype=np.float64) if with_absv else None
    ap = absv.ctypes.data if with_absv else None
    qs, ks, vs = _strides(q), _strides(k), _strides(v)
    rc = lib.oracle_varlen_prefill(
        q.data_ptr(), qs.ctypes.data, k.data_ptr(), ks.ctypes.data, v.data_ptr(), vs.ctypes.data,
        cq.ctypes.data, ck.ctypes.data, B, Hq, Hkv, Dk, Dv, int(bool(causal)), float(scale),
        rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data, ap,
        int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_varlen_prefill failed with code {rc}")
    return (out, lse, absv) if with_absv else (out, lse)
