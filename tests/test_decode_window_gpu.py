"""Sliding-window paged decode on the GPU, through the C ABI, against the fp64
oracle ("TokenSpeed-MLA 2.0.1", window_left: token t of a row with n keys sees
keys max(0, n - q_len + t - W) .. n - q_len + t).

BF16 and FP8 E4M3 caches; windows of 0, 1, around the 128-key tile and wider
than the rows; q_len 1-4; page sizes 16-256; forced split-KV chunking; pages
wholly before the window evicted (table entries -1, contents NaN), which the
kernels must neither look up nor load; head groupings of 16 and 32 rows and
head dim 256; argument checks; the full-size Qwen3-14B-shaped workload with a
4096-key window on sampled rows; repeated launches bitwise identical.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, DecodeWorkload, make_decode_inputs
from tests.gpu_common import BF16_UNIT, FP16_UNIT, built_library, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    yield lib
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def wl_window(lens, q_len=1, hq=8, hkv=2, ps=16, d=128, fp8=False, seed=61):
    return DecodeWorkload("win", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim_qk=d, head_dim_v=d, page_size=ps, scale=1.0 / math.sqrt(d),
                          seq_lens=tuple(lens), kv_fp8=fp8, value_seed=seed, spare_pages=3)


def evict_before_window(inp, wl, window):
    """Pages wholly before a row's first visible key: NaN contents, table entry -1."""
    bt = inp["block_table"].clone()
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    fp8 = kc.dtype == torch.float8_e4m3fn
    for b in range(wl.batch):
        n = int(inp["seq_lens"][b])
        first = max(0, n - wl.q_len - window)
        for pg in range(first // wl.page_size):
            phys = int(bt[b, pg])
            if fp8:
                kc.view(torch.uint8)[phys] = 0x7F
                vc.view(torch.uint8)[phys] = 0x7F
            else:
                kc[phys] = float("nan")
                vc[phys] = float("nan")
            bt[b, pg] = -1
    inp = dict(inp)
    inp["block_table"], inp["k_cache"], inp["v_cache"] = bt, kc, vc
    return inp


def run_case(fw, wl, window, chunk=0, evict=False, mapping="random"):
    inp = make_decode_inputs(wl, "cpu", mapping=mapping)
    if evict:
        inp = evict_before_window(inp, wl, window)
    ks = inp.get("k_scale", 1.0) if wl.kv_fp8 else 1.0
    vs = inp.get("v_scale", 1.0) if wl.kv_fp8 else 1.0
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], k_scale=ks, v_scale=vs, window_left=window, with_absv=True)
    d = to_device(inp)
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode_window(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                          d["scale"], window, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    assert fw.device_status() == 0
    return compare(out, lse, ref_o, ref_l,
                   what=f"window {window} fp8={wl.kv_fp8} {wl.seq_lens} q_len={wl.q_len} ps={wl.page_size}", absv=ref_a,
                   p_unit=FP16_UNIT if wl.kv_fp8 else BF16_UNIT)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("window", [0, 1, 7, 127, 128, 129, 300, 5000])
def test_window_sizes(fw, fp8, window):
    run_case(fw, wl_window([1, 130, 700, 1029, 2000], fp8=fp8), window)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("q_len", [2, 3, 4])
def test_multi_token_rows(fw, fp8, q_len):
    """Each query token has its own window; the first rows see fewer keys."""
    run_case(fw, wl_window([3, 129, 777], q_len=q_len, hq=8, hkv=2, fp8=fp8), 100)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("ps", [16, 64, 128, 256])
def test_page_sizes_with_evicted_pages(fw, fp8, ps):
    """Pages wholly before the window hold NaN and have table entries of -1:
    the kernels must neither look them up nor let them reach the MMAs."""
    run_case(fw, wl_window([300, 1029, 2222], q_len=2, ps=ps, fp8=fp8), 200, evict=True)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("chunk", [128, 512])
def test_forced_splits(fw, fp8, chunk):
    run_case(fw, wl_window([3000, 129, 5000], q_len=2, fp8=fp8), 1500, chunk=chunk)


@pytest.mark.parametrize("hq,hkv,q_len,d", [(40, 8, 1, 128), (64, 8, 4, 128), (96, 1, 1, 128), (16, 2, 2, 256)])
def test_head_groupings_bf16(fw, hq, hkv, q_len, d):
    run_case(fw, wl_window([400, 1500], q_len=q_len, hq=hq, hkv=hkv, d=d), 333)


@pytest.mark.parametrize("hq,hkv,q_len", [(40, 8, 1), (32, 8, 4), (96, 1, 1)])
def test_head_groupings_fp8(fw, hq, hkv, q_len):
    run_case(fw, wl_window([400, 1500], q_len=q_len, hq=hq, hkv=hkv, fp8=True), 333)


def test_no_window_equals_plain_decode(fw):
    wl = wl_window([37, 400, 1029], q_len=2)
    d = to_device(make_decode_inputs(wl, "cpu"))
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    o1, l1 = fw.paged_decode(*args)
    o2, l2 = fw.paged_decode_window(*args, -1)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_invalid_window_arguments_launch_nothing(fw):
    wl = wl_window([100])
    d = to_device(make_decode_inputs(wl, "cpu"))
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    before = fw.launch_count()
    with pytest.raises(fw.FwError):
        fw.paged_decode_window(*args, -2)
    with pytest.raises(fw.FwError):                       # scales apply to FP8 caches only
        fw.paged_decode_window(*args, 10, k_scale=2.0)
    assert fw.launch_count() == before


@pytest.mark.parametrize("fp8", [False, True])
def test_qwen3_14b_window_4096_full_size_sampled_rows(fw, fp8):
    """64 x (40/8 heads) x 128-token pages, lengths 512-32768, a 4096-key window,
    in the launch configuration the benchmark times; 48 sampled rows."""
    wl = WORKLOADS["qwen3_14b_paged_decode_fp8" if fp8 else "qwen3_14b_paged_decode"]
    W = 4096
    d = make_decode_inputs(wl, "cuda")
    ks, vs = (d["k_scale"], d["v_scale"]) if fp8 else (1.0, 1.0)
    out, lse = fw.paged_decode_window(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                      d["scale"], W, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    g = torch.Generator().manual_seed(7)
    lens = d["seq_lens"].cpu()
    bt = d["block_table"].cpu()
    for b in torch.randperm(wl.batch, generator=g)[:12].tolist():
        npg = -(-int(lens[b]) // wl.page_size)
        pages = bt[b, :npg].long()
        if fp8:
            k = d["k_cache"].view(torch.uint8)[pages.cuda()].cpu().view(torch.float8_e4m3fn)
            v = d["v_cache"].view(torch.uint8)[pages.cuda()].cpu().view(torch.float8_e4m3fn)
        else:
            k = d["k_cache"][pages.cuda()].cpu()
            v = d["v_cache"][pages.cuda()].cpu()
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        heads = torch.randperm(wl.num_q_heads, generator=g)[:4].tolist()
        o_ref, l_ref, a_ref = oracle.paged_decode(d["q"][b:b + 1].cpu(), k, v, sub_bt, lens[b:b + 1], wl.scale,
                                                  rows=heads, k_scale=ks, v_scale=vs, window_left=W, with_absv=True)
        compare(out[b, 0, heads], lse[b, 0, heads], o_ref, l_ref, f"b{b}", absv=a_ref,
                p_unit=FP16_UNIT if fp8 else BF16_UNIT)


@pytest.mark.parametrize("fp8", [False, True])
def test_repeated_window_launches_are_bitwise_identical(fw, fp8):
    wl = WORKLOADS["qwen3_14b_paged_decode_fp8" if fp8 else "qwen3_14b_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    ks, vs = (d["k_scale"], d["v_scale"]) if fp8 else (1.0, 1.0)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"], 4096)
    out0, lse0 = fw.paged_decode_window(*args, k_scale=ks, v_scale=vs)
    for _ in range(3):
        out, lse = fw.paged_decode_window(*args, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))
