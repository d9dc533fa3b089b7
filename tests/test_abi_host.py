"""Host-side checks of the C ABI that need no GPU.

  * libfw_attn.so builds, loads and exports every function include/*.h declares;
  * the decode planner's folding, split sizing and workspace size agree with
    the pages' formulas as restated independently in oracle/planning.py;
  * invalid arguments are rejected with the documented status before any
    CUDA call, and a valid call without a usable GPU fails loudly.
"""
import ctypes
import glob
import os
import re

import pytest

from oracle import planning

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fwlib():
    from ragged_softmax_attention_gb300 import build
    import ragged_softmax_attention_gb300 as fw
    path = build.build()
    fw.load_library(path)
    return fw


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(fw_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fw_paged_decode", "fw_varlen_prefill", "fw_paged_decode_workspace_size",
                     "fw_set_workspace", "fw_get_device_status", "fw_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(fwlib):
    lib = ctypes.CDLL(fwlib._binding.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_missing_library_fails_loudly():
    from ragged_softmax_attention_gb300 import _binding
    saved = _binding._lib
    _binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            _binding.load_library("/nonexistent/libfw_attn.so")
    finally:
        _binding._lib = saved


@pytest.mark.parametrize("G,q_len", [(5, 1), (4, 1), (8, 4), (5, 4), (16, 4), (12, 4), (32, 2), (3, 3), (1, 4)])
def test_planner_folds_like_tokenspeed_rule(fwlib, G, q_len):
    p = fwlib.plan_decode(2, q_len, G * 2, 2, 128, 4096, num_sms=152)
    F = planning.fold_factor(G, q_len, max_rows=32)
    assert p["tokens_per_unit"] == F
    assert p["row_groups"] == q_len // F
    assert p["rows_per_unit"] == (16 if G * F <= 16 else 32)


def test_planner_wide_groups_are_chunked(fwlib):
    p = fwlib.plan_decode(2, 4, 128, 1, 128, 81920, num_sms=152)
    assert p["heads_per_unit"] == 32 and p["row_groups"] == 4 * 4


@pytest.mark.parametrize("q_len,hq,hkv,sms,grid", [(4, 128, 1, 152, 152), (3, 128, 1, 152, 150),
                                                    (1, 64, 1, 152, 152), (2, 128, 2, 148, 148)])
def test_planner_latent_row_groups_ride_on_the_grid(fwlib, q_len, hq, hkv, sms, grid):
    """Latent heads (Dv 512): a row group is 128 heads of one token on a CTA
    pair when the group holds a multiple of 128 heads, else 64 heads on one
    CTA; the row groups of a unit are consecutive workers, so the grid is a
    whole multiple of them (two CTAs per pair)."""
    p = fwlib.plan_decode(32, q_len, hq, hkv, 512, 81920, num_sms=sms)
    G = hq // hkv
    rows = 128 if G % 128 == 0 else 64
    assert p["heads_per_unit"] == rows and p["rows_per_unit"] == rows and p["tokens_per_unit"] == 1
    assert p["row_groups"] == q_len * G // rows
    per = p["row_groups"] * (2 if rows == 128 else 1)
    assert p["grid"] == grid and p["grid"] % per == 0
    assert p["min_span_tiles"] == 32
    assert p["max_pieces"] == -(-640 // 32) + 1


def test_planner_latent_rejects_partial_head_blocks(fwlib):
    """Several KV heads: a row group holds one token's heads, so 48 heads per
    KV head (not a multiple of 64) cannot be served."""
    with pytest.raises(fwlib.FwError):
        fwlib.plan_decode(2, 1, 96, 2, 512, 4096, num_sms=152)


@pytest.mark.parametrize("hq,q_len", [(96, 4), (96, 8), (128, 4), (64, 2), (48, 3), (16, 4), (16, 1), (32, 3)])
def test_planner_latent_packed_rows(fwlib, hq, q_len):
    """One KV head: query rows are packed as token * H + head ("TokenSpeed-MLA
    2.0.1", packed-query paragraph).  At 128 or more rows the groups are the
    pages' 128-row query tiles, ceil(H * q_len / 128) of them (H96/Sq4 -> 3,
    H96/Sq8 -> 6), on CTA pairs; fewer rows make 64-row groups on one CTA."""
    p = fwlib.plan_decode(4, q_len, hq, 1, 512, 8192, num_sms=152)
    if hq * q_len >= 128:
        assert p["rows_per_unit"] == 128
        assert p["row_groups"] == planning.packed_q_tiles(hq, q_len)
        assert p["grid"] % (2 * p["row_groups"]) == 0
    else:
        assert p["rows_per_unit"] == 64 and p["row_groups"] == -(-hq * q_len // 64)


def test_planner_workspace_matches_pages_formula(fwlib):
    """Dv + 1 FP32 values per row per split: at H*q_len a multiple of 128 the
    partials take exactly TokenSpeed's B*128*ceil(H*q_len/128)*split*513*4 bytes."""
    p = fwlib.plan_decode(2, 4, 128, 1, 512, 81920, num_sms=152)
    assert p["max_pieces"] > 1
    assert p["partial_bytes"] == planning.split_workspace_bytes(2, 128, 4, p["max_pieces"], 512)
    assert p["workspace_bytes"] >= p["partial_bytes"] + (2 + 3) * 4
    p1 = fwlib.plan_decode(2, 1, 8, 2, 128, 200, num_sms=152)
    assert p1["partial_bytes"] == 2 * 8 * p1["max_pieces"] * 129 * 4


def test_planner_piece_bound(fwlib):
    """A unit of t tiles meets at most ceil(t / span) + 1 CTA ranges."""
    for max_len in (1, 127, 128, 129, 4096, 32768, 81920):
        p = fwlib.plan_decode(64, 1, 40, 8, 128, max_len, num_sms=152)
        tiles = -(-max_len // 128)
        assert p["min_span_tiles"] == 8
        assert p["max_pieces"] == -(-tiles // 8) + 1
        assert p["num_units"] == 64 * 8 * p["row_groups"]
        assert p["grid"] == 152


def piece_count(start, tiles, span):
    """Ranges [r*span, (r+1)*span) that tiles [start, start + tiles) meet."""
    return len({t // span for t in range(start, start + tiles)})


def test_piece_bound_holds_for_any_alignment():
    for span in (1, 3, 8, 100):
        for tiles in (1, 2, 7, 8, 9, 64, 257):
            worst = max(piece_count(s, tiles, span) for s in range(span))
            assert worst <= -(-tiles // span) + 1


def test_qwen3_14b_plan(fwlib):
    """40 Q / 8 KV heads, q_len 1: one unit holds the five query heads of a KV
    head (PyPTO section 1.3), padded to a 16-row MMA N extent."""
    p = fwlib.plan_decode(64, 1, 40, 8, 128, 32768, num_sms=152)
    assert p["group"] == 5 and p["heads_per_unit"] == 5 and p["rows_per_unit"] == 16
    assert p["row_groups"] == 1


def test_forced_chunk_option(fwlib):
    fwlib.set_option(fwlib.FW_OPT_DECODE_CHUNK_TOKENS, 256)
    try:
        p = fwlib.plan_decode(2, 1, 8, 2, 128, 1000, num_sms=152)
        assert p["min_span_tiles"] == 2 and p["max_pieces"] == 4 + 1
    finally:
        fwlib.set_option(fwlib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    with pytest.raises(fwlib.FwError):
        fwlib.set_option(fwlib.FW_OPT_DECODE_CHUNK_TOKENS, 100)


def test_prefill_softmax_option(fwlib):
    """0 (static anchor) and 1 (online, conditional rescale) are the only modes."""
    for mode in (1, 0):
        fwlib.set_option(fwlib.FW_OPT_PREFILL_SOFTMAX, mode)
    for bad in (-1, 2):
        with pytest.raises(fwlib.FwError):
            fwlib.set_option(fwlib.FW_OPT_PREFILL_SOFTMAX, bad)


# ------------------------------------------------------- validation, no GPU

def fake(shape, dtype, ptr=0x10000, strides=None):
    from ragged_softmax_attention_gb300._binding import FwTensor
    t = FwTensor()
    t.data = ptr
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides = []
        acc = 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        t.shape[i] = s
        t.stride[i] = st
    return t


def call_decode(fwlib, q, k, v, bt, sl, out, lse=None, scale=0.1):
    lib = fwlib.load_library()
    r = lambda x: ctypes.byref(x) if x is not None else None
    return lib.fw_paged_decode(r(q), r(k), r(v), r(bt), r(sl), ctypes.c_float(scale), r(out), r(lse), None)


def decode_args(B=2, q_len=1, Hq=8, Hkv=2, D=128, P=10, ps=16, max_pages=4):
    BF, F32, I32 = 0, 1, 2
    return dict(q=fake([B, q_len, Hq, D], BF), k=fake([P, ps, Hkv, D], BF), v=fake([P, ps, Hkv, D], BF),
                bt=fake([B, max_pages], I32), sl=fake([B], I32), out=fake([B, q_len, Hq, D], BF),
                lse=fake([B, q_len, Hq], F32))


@pytest.mark.parametrize("mutate,status", [
    (lambda a: a["q"].__setattr__("dtype", 1), 1),                 # q not bf16
    (lambda a: a["k"].__setattr__("ndim", 3), 1),                  # wrong rank
    (lambda a: a["out"].shape.__setitem__(3, 64), 1),              # out head dim mismatch
    (lambda a: a["sl"].shape.__setitem__(0, 3), 1),                # seq_lens length
    (lambda a: a["q"].__setattr__("data", 0x10002), 1),            # misaligned base
    (lambda a: a["k"].stride.__setitem__(1, 2 * 128 + 4), 1),      # stride not 16-byte multiple
    (lambda a: a["bt"].stride.__setitem__(1, 2), 1),               # non-contiguous table rows
    (lambda a: a["lse"].shape.__setitem__(2, 5), 1),               # lse shape
])
def test_invalid_decode_arguments(fwlib, mutate, status):
    a = decode_args()
    mutate(a)
    rc = call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"])
    assert rc == status, fwlib.load_library().fw_last_error()


def test_unsupported_shapes(fwlib):
    a = decode_args(D=64)
    assert call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"]) == 2
    a = decode_args(ps=24)
    assert call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"]) == 2
    a = decode_args(q_len=5)
    assert call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"]) == 2
    a = decode_args(Hq=6, Hkv=4)
    assert call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"]) == 1


def test_nonfinite_scale_rejected(fwlib):
    a = decode_args()
    assert call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"],
                       scale=float("nan")) == 1


def test_valid_call_without_gpu_fails_loudly(fwlib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = decode_args()
    rc = call_decode(fwlib, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["out"], a["lse"])
    assert rc in (2, 4)              # FW_ERR_UNSUPPORTED / FW_ERR_CUDA: no device, nothing launched
    assert fwlib.launch_count() == 0
