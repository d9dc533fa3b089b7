"""Latent-head paged decode (Dk 576, Dv 512) on the GPU, through the C ABI,
against the fp64 oracle.

The layout of "TokenSpeed-MLA 2.0.1" (decode): one KV head whose 576-wide rows
are the keys and whose first 512 columns are the values, 128 query heads, up
to four query tokens with bottom-right causal rows.  Covers ragged lengths
around tile and page boundaries (NaN-poisoned slots past each row's end),
rows that see no key, q_len 1-4, 64-head groups and two KV heads, packed
(token, head) rows for head counts that are not a multiple of 64, sliding
windows with evicted pages, page sizes
16-256, forced split-KV chunking, score scales large enough to move the
static anchors, a separate (non-aliased) value cache, and the full-size
workload on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, DecodeWorkload, make_decode_inputs
from tests.gpu_common import built_library, compare, to_device
from tests.test_decode_window_gpu import evict_before_window

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    yield lib
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def wl_latent(lens, q_len=4, hq=128, hkv=1, ps=64, scale=0.07216882, seed=21, aliased=True):
    return DecodeWorkload("latent", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim_qk=576, head_dim_v=512, page_size=ps, scale=scale,
                          seq_lens=tuple(lens), latent=aliased, value_seed=seed, spare_pages=3)


def run_case(fw, wl, chunk=0, mapping="random"):
    inp = make_decode_inputs(wl, "cpu", mapping=mapping)
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], with_absv=True)
    d = to_device(inp)
    if wl.latent:
        d["v_cache"] = d["k_cache"][..., :512]
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                   d["scale"])
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    assert fw.device_status() == 0
    return compare(out, lse, ref_o, ref_l, what=f"latent {wl.seq_lens} q_len={wl.q_len} ps={wl.page_size}", absv=ref_a)


def test_ragged_lengths_around_tiles_and_pages(fw):
    """Lengths 1..5 (fewer keys than query tokens: those rows see nothing),
    63/64/65 (page), 127/128/129 (tile), and a multi-tile tail."""
    run_case(fw, wl_latent([1, 2, 3, 4, 5, 63, 64, 65, 127, 128, 129, 700]))


@pytest.mark.parametrize("q_len", [1, 2, 3])
def test_query_token_counts(fw, q_len):
    run_case(fw, wl_latent([300, 1000], q_len=q_len))


@pytest.mark.parametrize("hq,hkv", [(64, 1), (128, 2)])
def test_head_groups_of_64(fw, hq, hkv):
    run_case(fw, wl_latent([200, 513], hq=hq, hkv=hkv))


@pytest.mark.parametrize("ps", [16, 32, 128, 256])
def test_page_sizes(fw, ps):
    run_case(fw, wl_latent([37, 400, 1029], ps=ps))


@pytest.mark.parametrize("mapping", ["identity", "reverse", "shared_prefix"])
def test_adversarial_block_tables(fw, mapping):
    run_case(fw, wl_latent([640, 900], q_len=2), mapping=mapping)


@pytest.mark.parametrize("chunk", [128, 512, 4096])
def test_forced_splits(fw, chunk):
    """Many pieces per unit: partials merged by the combine kernel."""
    run_case(fw, wl_latent([3000, 129, 5000], q_len=2), chunk=chunk)


def test_empty_rows(fw):
    run_case(fw, wl_latent([0, 150, 0], q_len=3))


@pytest.mark.parametrize("scale", [4.0, -2.0])
def test_scales_that_move_the_anchor(fw, scale):
    """Scores spread over hundreds of log2 units: later tiles rise far above
    the first tile's maxima, so anchors move and O^T is rescaled in TMEM."""
    fw.read_counters()                                   # reset
    run_case(fw, wl_latent([2000, 1300], q_len=2, scale=scale, seed=23))
    assert fw.read_counters()["latent_rescales"] > 0, "no anchor moved"


@pytest.mark.parametrize("hq,q_len", [(16, 4), (16, 1), (96, 4), (64, 2), (48, 3), (32, 4)])
def test_packed_query_rows(fw, hq, q_len):
    """Head counts that are not a multiple of the row group: rows packed as
    token * H + head, so a row group straddles tokens (each row keeps its own
    causal bound) and the last group is padded.  Short rows (1-5 keys) make
    whole tokens see nothing."""
    run_case(fw, wl_latent([1, 3, 5, 130, 700], q_len=q_len, hq=hq, seed=27))


@pytest.mark.parametrize("chunk", [128, 1024])
def test_packed_query_rows_with_splits(fw, chunk):
    """Packed rows (H96, q_len 4: three 128-row groups) with many split-KV
    pieces merged by the combine kernel."""
    run_case(fw, wl_latent([3000, 257, 1800], q_len=4, hq=96, seed=29), chunk=chunk)


def run_window_case(fw, wl, window, chunk=0):
    """Sliding window ("TokenSpeed-MLA 2.0.1", window_left, defined there for
    this layout); pages wholly before a row's window are evicted (NaN, table
    entry -1), so touching one shows up as NaN or a bad-page status."""
    inp = evict_before_window(make_decode_inputs(wl, "cpu"), wl, window)
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], window_left=window, with_absv=True)
    d = to_device(inp)
    if wl.latent:
        d["v_cache"] = d["k_cache"][..., :512]
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode_window(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                          d["scale"], window)
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    assert fw.device_status() == 0
    return compare(out, lse, ref_o, ref_l, what=f"latent window {window} {wl.seq_lens} q_len={wl.q_len} H={wl.num_q_heads}", absv=ref_a)


@pytest.mark.parametrize("window", [0, 1, 100, 127, 128, 129, 300, 5000])
def test_window_sizes(fw, window):
    """CTA pairs, 128 heads, q_len 4: each token's window starts one key later."""
    run_window_case(fw, wl_latent([1, 5, 130, 700, 2000], q_len=4), window)


@pytest.mark.parametrize("hq,hkv,q_len,ps,window", [(96, 1, 4, 16, 100), (16, 1, 4, 32, 50), (128, 2, 2, 32, 129),
                                                    (48, 1, 3, 64, 200)])
def test_window_packed_rows_and_one_cta(fw, hq, hkv, q_len, ps, window):
    """Packed rows (a group's rows have different windows), the one-CTA kernel,
    and pages smaller than a tile (leading pages of the first tile skipped)."""
    run_window_case(fw, wl_latent([3, 129, 777, 1500], q_len=q_len, hq=hq, hkv=hkv, ps=ps, seed=31), window)


def test_window_with_splits(fw):
    """A 1000-key window over long rows, cut into many split-KV pieces."""
    run_window_case(fw, wl_latent([4000, 2600, 1100], q_len=2, seed=33), 1000, chunk=512)


def test_separate_value_cache(fw):
    """Dv = 512 values from their own cache instead of a view of the keys."""
    run_case(fw, wl_latent([333, 1200], q_len=2, aliased=False, seed=25))


def test_latent_workload_full_size_sampled_rows(fw):
    """32 rows x 81920 keys, 128/1 heads, q_len 4, pages of 64, in the launch
    configuration the benchmark times; 64 sampled rows against the oracle and
    every output finite."""
    wl = WORKLOADS["latent_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    g = np.random.default_rng(13)
    lens = d["seq_lens"].cpu()
    bt = d["block_table"].cpu()
    for b in g.choice(wl.batch, size=4, replace=False).tolist():
        npg = -(-int(lens[b]) // wl.page_size)
        pages = bt[b, :npg].long()
        k = d["k_cache"][pages.cuda()].cpu()
        v = k[..., :wl.head_dim_v]
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        t = g.integers(0, wl.q_len, size=16)
        h = g.choice(wl.num_q_heads, size=16, replace=False)
        rows = (t * wl.num_q_heads + h).tolist()
        o_ref, l_ref, a_ref = oracle.paged_decode(d["q"][b:b + 1].cpu(), k, v, sub_bt, lens[b:b + 1], wl.scale, rows=rows, with_absv=True)
        tt, hh = torch.as_tensor(t, device="cuda"), torch.as_tensor(h, device="cuda")
        compare(out[b, tt, hh], lse[b, tt, hh], o_ref, l_ref, f"b{b}", absv=a_ref)


def test_invalid_latent_shapes_launch_nothing(fw):
    wl = wl_latent([100], hq=128)
    d = to_device(make_decode_inputs(wl, "cpu"))
    before = fw.launch_count()
    with pytest.raises(fw.FwError):                     # 96 of 128 heads: q not one stride over (token, head)
        fw.paged_decode(d["q"][:, :, :96], d["k_cache"], d["k_cache"][..., :512], d["block_table"],
                        d["seq_lens"], 0.1)
    with pytest.raises(fw.FwError):                     # Dv 512 with Dk 512: not the latent layout
        fw.paged_decode(d["q"][..., :512], d["k_cache"][..., :512], d["k_cache"][..., :512], d["block_table"],
                        d["seq_lens"], 0.1)
    assert fw.launch_count() == before


def test_repeated_launches_are_bitwise_identical(fw):
    """Every launch writes the same bytes (an accumulator read before its last
    MMA has landed shows up as drift between launches).  Full-size latent
    workload, four launches."""
    wl = WORKLOADS["latent_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    out0, lse0 = fw.paged_decode(*args)
    for _ in range(3):
        out, lse = fw.paged_decode(*args)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))
