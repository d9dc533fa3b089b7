"""Paged decode over an FP8 E4M3 KV cache on the GPU, through the C ABI,
against the fp64 oracle on the same bytes and scales.

"TokenSpeed-MLA 2.0.1" (decode: FP8 inputs, BF16 output).  The oracle takes
k = k_scale * e4m3(byte), v = v_scale * e4m3(byte) exactly, so the parity bar
is the BF16 path's.  Covers lengths around tile and page boundaries with
NaN bytes in unused slots, page sizes 8-256, query-head groupings that fold
to 16 and 32 rows, causal multi-token rows, forced split-KV chunking, empty
rows, adversarial block tables, scale handling, argument checks and the
full-size Qwen3-14B-shaped workload on sampled rows.
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


def wl_fp8(lens, q_len=1, hq=8, hkv=2, ps=16, seed=51):
    return DecodeWorkload("fp8", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim_qk=128, head_dim_v=128, page_size=ps, scale=1.0 / math.sqrt(128),
                          seq_lens=tuple(lens), kv_fp8=True, value_seed=seed, spare_pages=3)


def run_case(fw, wl, chunk=0, mapping="random", k_scale=None, v_scale=None):
    inp = make_decode_inputs(wl, "cpu", mapping=mapping)
    ks = inp["k_scale"] if k_scale is None else k_scale
    vs = inp["v_scale"] if v_scale is None else v_scale
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], k_scale=ks, v_scale=vs, with_absv=True)
    d = to_device(inp)
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                       d["scale"], ks, vs)
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    assert fw.device_status() == 0
    return compare(out, lse, ref_o, ref_l, what=f"fp8 {wl.seq_lens} q_len={wl.q_len} ps={wl.page_size}", absv=ref_a, p_unit=FP16_UNIT)


def test_tiny_fp8_decode(fw):
    run_case(fw, wl_fp8([37, 200]))


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 511, 700])
def test_boundary_lengths(fw, n):
    run_case(fw, wl_fp8([n, 5]))


@pytest.mark.parametrize("ps", [8, 16, 32, 64, 128, 256])
def test_page_sizes(fw, ps):
    run_case(fw, wl_fp8([37, 300, 1029], ps=ps))


@pytest.mark.parametrize("hq,hkv,q_len", [(40, 8, 1), (32, 8, 4), (64, 8, 4), (96, 1, 1), (8, 8, 2)])
def test_head_groupings(fw, hq, hkv, q_len):
    """Folded query rows of 16 (5, 4x4, 2x1 heads) and 32 (8x4 heads, 96 heads in 32-head chunks)."""
    run_case(fw, wl_fp8([130, 333], q_len=q_len, hq=hq, hkv=hkv))


@pytest.mark.parametrize("chunk", [128, 512])
def test_forced_splits(fw, chunk):
    run_case(fw, wl_fp8([2000, 129, 3000], q_len=2), chunk=chunk)


def test_empty_rows(fw):
    run_case(fw, wl_fp8([0, 150, 0], q_len=3))


@pytest.mark.parametrize("mapping", ["identity", "reverse", "shared_prefix"])
def test_adversarial_block_tables(fw, mapping):
    run_case(fw, wl_fp8([640, 900]), mapping=mapping)


def test_scales_are_applied(fw):
    """Scales other than the generator's (about 0.01 each): k_scale doubles the
    scores' spread, v_scale doubles the output; outputs stay of order 1, where
    the stated absolute bar is meaningful for BF16."""
    run_case(fw, wl_fp8([400, 77]), k_scale=0.02, v_scale=0.02)


def test_invalid_fp8_arguments_launch_nothing(fw):
    wl = wl_fp8([100])
    d = to_device(make_decode_inputs(wl, "cpu"))
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    before = fw.launch_count()
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0)):
        with pytest.raises(fw.FwError):
            fw.paged_decode_fp8(*args, ks, vs)
    with pytest.raises(fw.FwError):                      # FP8 caches through the BF16 entry point
        fw.paged_decode(*args)
    bf = d["k_cache"].to(torch.bfloat16)
    with pytest.raises(fw.FwError):                      # BF16 caches through the FP8 entry point
        fw.paged_decode_fp8(d["q"], bf, bf, d["block_table"], d["seq_lens"], d["scale"], 1.0, 1.0)
    assert fw.launch_count() == before


def test_qwen3_14b_fp8_decode_full_size_sampled_rows(fw):
    """64 x (40/8 heads) x 128-token pages at full size in the benchmark's launch
    configuration; 48 sampled (b, h) rows against the oracle, all outputs finite."""
    wl = WORKLOADS["qwen3_14b_paged_decode_fp8"]
    d = make_decode_inputs(wl, "cuda")
    out, lse = fw.paged_decode_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                   d["scale"], d["k_scale"], d["v_scale"])
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    g = torch.Generator().manual_seed(5)
    bs = torch.randperm(wl.batch, generator=g)[:12].tolist()
    lens = d["seq_lens"].cpu()
    bt = d["block_table"].cpu()
    for b in bs:
        npg = -(-int(lens[b]) // wl.page_size)
        pages = bt[b, :npg].long()
        k = d["k_cache"].view(torch.uint8)[pages.cuda()].cpu().view(torch.float8_e4m3fn)
        v = d["v_cache"].view(torch.uint8)[pages.cuda()].cpu().view(torch.float8_e4m3fn)
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        heads = torch.randperm(wl.num_q_heads, generator=g)[:4].tolist()
        o_ref, l_ref, a_ref = oracle.paged_decode(d["q"][b:b + 1].cpu(), k, v, sub_bt, lens[b:b + 1], wl.scale,
                                                  rows=heads, k_scale=d["k_scale"], v_scale=d["v_scale"], with_absv=True)
        compare(out[b, 0, heads], lse[b, 0, heads], o_ref, l_ref, f"b{b}", absv=a_ref, p_unit=FP16_UNIT)


@pytest.mark.parametrize("chunk", [0, 512])
def test_repeated_launches_are_bitwise_identical(fw, chunk):
    """Every launch writes the same bytes (an accumulator read before its last
    MMA has landed shows up as drift between launches).  Full-size FP8
    workload, six launches, with and without forced split-KV chunking."""
    wl = WORKLOADS["qwen3_14b_paged_decode_fp8"]
    d = make_decode_inputs(wl, "cuda")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"], d["k_scale"],
            d["v_scale"])
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out0, lse0 = fw.paged_decode_fp8(*args)
        for _ in range(5):
            out, lse = fw.paged_decode_fp8(*args)
            torch.cuda.synchronize()
            assert fw.device_status() == 0
            assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
