"""Paged decode on the GPU, through the C ABI, against the fp64 oracle.

Covers the boundary matrix of "Writing Page Attention with PyPTO", section
10.1 (seq_len 1, page and 512-token stack boundaries, 1/2/3-page tails, a
ragged batch), its adversarial block tables (section 10.2: random, reverse,
shared-prefix), NaN-poisoned unused pages and tail slots (a read outside the
ragged extent poisons the output), forced split-KV chunking vs. one pass,
q_len up to 4 with bottom-right causal rows, empty rows, guard zones around
the output, and the full-size Qwen3-14B-shaped workload on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, DecodeWorkload, make_decode_inputs
from tests.gpu_common import OUT_TOL, built_library, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    yield lib
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def run_case(fw, wl, lens=None, mapping="random", chunk=0, check_status=True):
    inp = make_decode_inputs(wl, "cpu", seq_lens=lens, mapping=mapping)
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], with_absv=True)
    d = to_device(inp)
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                   d["scale"])
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    if check_status:
        assert fw.device_status() == 0
    return compare(out, lse, ref_o, ref_l, what=wl.name, absv=ref_a), out, lse


def wl_decode(batch=3, q_len=1, hq=8, hkv=2, d=128, ps=16, lens=(37, 200, 5), seed=11, name="case"):
    return DecodeWorkload(name, batch=batch, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim_qk=d, head_dim_v=d, page_size=ps, scale=1.0 / math.sqrt(d),
                          seq_lens=tuple(lens), value_seed=seed, spare_pages=4)


def test_tiny_paged_decode_workload(fw):
    """The tiny workload exactly as specified: B=2, 8/2 heads, hd 128, ps 16, n = [37, 200]."""
    (err, lerr), _, _ = run_case(fw, WORKLOADS["tiny_paged_decode"])
    assert err <= OUT_TOL and lerr <= 1e-3


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 511, 512, 513, 700])
def test_boundary_lengths(fw, n):
    run_case(fw, wl_decode(batch=2, lens=(n, max(1, n // 3)), ps=128, hq=40, hkv=8, name=f"n{n}"))


@pytest.mark.parametrize("ps", [8, 16, 32, 64, 128, 256])
def test_page_sizes_and_tails(fw, ps):
    # 1/2/3-page tails and a ragged batch for every supported page size
    lens = (ps + 1, 2 * ps + 3, 3 * ps - 1, 5)
    run_case(fw, wl_decode(batch=4, ps=ps, lens=lens, name=f"ps{ps}"))


@pytest.mark.parametrize("mapping", ["random", "reverse", "identity", "shared_prefix"])
def test_adversarial_block_tables(fw, mapping):
    run_case(fw, wl_decode(batch=4, ps=16, lens=(300, 41, 97, 260)), mapping=mapping)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (40, 8), (16, 2), (32, 4), (64, 2), (64, 1), (96, 1)])
def test_gqa_groups(fw, hq, hkv):
    run_case(fw, wl_decode(batch=2, hq=hq, hkv=hkv, ps=64, lens=(517, 90)))


@pytest.mark.parametrize("q_len", [2, 3, 4])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (40, 8), (16, 1), (12, 1), (64, 1)])
def test_multi_token_causal(fw, q_len, hq, hkv):
    run_case(fw, wl_decode(batch=3, q_len=q_len, hq=hq, hkv=hkv, ps=32, lens=(3, 300, 129)))


def test_head_dim_256(fw):
    run_case(fw, wl_decode(batch=3, d=256, hq=16, hkv=2, ps=64, lens=(700, 129, 1)))


@pytest.mark.parametrize("chunk", [128, 256, 1024])
def test_forced_splits_match_oracle(fw, chunk):
    run_case(fw, wl_decode(batch=3, hq=40, hkv=8, ps=128, lens=(2000, 513, 127)), chunk=chunk)


def test_split_count_invariance(fw):
    """Different split chunkings agree with each other to rounding (not bitwise)."""
    wl = wl_decode(batch=2, hq=40, hkv=8, ps=64, lens=(3000, 1500))
    outs = []
    for chunk in (0, 128, 384, 2048):
        _, out, lse = run_case(fw, wl, chunk=chunk)
        outs.append((out.float().cpu(), lse.cpu()))
    for o, l in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= OUT_TOL
        assert (l - outs[0][1]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("scale", [1.0, -0.2])
def test_scale_extremes_exercise_rescale(fw, scale):
    """Large or negative scales move the running max far and often."""
    wl = wl_decode(batch=3, hq=40, hkv=8, ps=64, lens=(900, 130, 2000))
    import dataclasses
    run_case(fw, dataclasses.replace(wl, scale=scale), chunk=256)


def test_empty_rows(fw):
    """n = 0 rows and causal rows with no visible key: zero output, -inf LSE."""
    run_case(fw, wl_decode(batch=3, q_len=4, lens=(0, 2, 40), ps=16))


def test_output_guard_zones(fw):
    wl = wl_decode(batch=2, hq=8, hkv=2, ps=16, lens=(100, 33))
    inp = to_device(make_decode_inputs(wl, "cpu"))
    big = torch.full((4, 1, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    big_lse = torch.full((4, 1, 8), 5.0, dtype=torch.float32, device="cuda")
    out, lse = fw.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                               inp["scale"], out=big[1:3], lse=big_lse[1:3])
    torch.cuda.synchronize()
    assert torch.all(big[0] == 7.0) and torch.all(big[3] == 7.0)
    assert torch.all(big_lse[0] == 5.0) and torch.all(big_lse[3] == 5.0)


def test_lse_optional(fw):
    wl = wl_decode(batch=2, lens=(77, 5))
    inp = make_decode_inputs(wl, "cpu")
    ref_o, _, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                          inp["seq_lens"], inp["scale"], with_absv=True)
    d = to_device(inp)
    out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"],
                               return_lse=False)
    assert lse is None
    compare(out, None, ref_o, None, "no-lse", absv=ref_a)


def test_invalid_arguments_launch_nothing(fw):
    wl = wl_decode(batch=2, lens=(77, 5))
    d = to_device(make_decode_inputs(wl, "cpu"))
    before = fw.launch_count()
    with pytest.raises(fw.FwError):                                   # wrong dtype
        fw.paged_decode(d["q"].float(), d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], 0.1)
    with pytest.raises(fw.FwError):                                   # Hq not a multiple of Hkv
        fw.paged_decode(d["q"][:, :, :7], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], 0.1)
    with pytest.raises(fw.FwError):                                   # unsupported head dim
        fw.paged_decode(d["q"][..., :64], d["k_cache"][..., :64], d["v_cache"][..., :64],
                        d["block_table"], d["seq_lens"], 0.1)
    assert fw.launch_count() == before


def test_qwen3_14b_decode_full_size_sampled_rows(fw):
    """The 64 x (40/8 heads) x 128-token-page workload at full size, in the launch
    configuration the benchmark times; 48 sampled (b, h) rows are checked
    against the oracle, and every output must be finite (NaN canaries)."""
    wl = WORKLOADS["qwen3_14b_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
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
        k = d["k_cache"][pages.cuda()].cpu()
        v = d["v_cache"][pages.cuda()].cpu()
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        heads = torch.randperm(wl.num_q_heads, generator=g)[:4].tolist()
        o_ref, l_ref, a_ref = oracle.paged_decode(d["q"][b:b + 1].cpu(), k, v, sub_bt, lens[b:b + 1], wl.scale,
                                                  rows=heads, with_absv=True)
        compare(out[b, 0, heads], lse[b, 0, heads], o_ref, l_ref, f"b{b}", absv=a_ref)


@pytest.mark.parametrize("chunk", [0, 512])
def test_repeated_launches_are_bitwise_identical(fw, chunk):
    """Every launch writes the same bytes.  An accumulator read before its last
    MMA has landed, or a buffer refilled while still in use, shows up as drift
    between launches.  Full-size Qwen3-14B-shaped workload, six launches, with
    and without forced split-KV chunking."""
    wl = WORKLOADS["qwen3_14b_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out0, lse0 = fw.paged_decode(*args)
        for _ in range(5):
            out, lse = fw.paged_decode(*args)
            torch.cuda.synchronize()
            assert fw.device_status() == 0
            assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
