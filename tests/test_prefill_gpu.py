"""Varlen prefill on the GPU, through the C ABI, against the fp64 oracle.

Ragged packs (TokenSpeed-MLA capability summary: no padding, Q and KV packs
may differ), causal bottom-right and non-causal, GQA and MHA, head dims 128
and 256, tile-boundary lengths, empty sequences and rows with no visible key,
and the two full-size workloads (varlen GQA prefill, dense causal MHA at head
dim 256) on sampled rows in the launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, PrefillWorkload, make_prefill_inputs
from tests.gpu_common import built_library, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    return built_library()


def wl_prefill(hq=8, hkv=2, d=128, causal=True, seed=31):
    return PrefillWorkload("p", num_seqs=0, num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=d, head_dim_v=d,
                           causal=causal, scale=1.0 / math.sqrt(d), value_seed=seed)


def run_case(fw, wl, lq, lk=None, rows=None):
    inp = make_prefill_inputs(wl, "cpu", lq, lk)
    ref_o, ref_l, ref_a = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                                wl.causal, wl.scale, rows=rows, with_absv=True)
    d = to_device(inp)
    out, lse = fw.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal, wl.scale)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    o = out.reshape(-1, out.shape[-1])
    l_ = lse.reshape(-1)
    if rows is not None:
        o, l_ = o[rows], l_[rows]
    return compare(o, l_, ref_o, ref_l, what=f"lq={lq} lk={lk}", absv=ref_a)


@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 257, 300, 511, 600])
def test_causal_single_sequence_lengths(fw, L):
    run_case(fw, wl_prefill(), [L])


@pytest.mark.parametrize("causal", [True, False])
def test_ragged_batch(fw, causal):
    run_case(fw, wl_prefill(causal=causal), [130, 1, 257, 64, 0, 400])


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 1), (32, 8), (12, 3)])
def test_gqa_groups(fw, hq, hkv):
    run_case(fw, wl_prefill(hq=hq, hkv=hkv), [200, 333])


@pytest.mark.parametrize("lq,lk", [([100, 5, 300], [500, 5, 300]), ([256, 40], [100, 40]), ([7, 129], [0, 600])])
@pytest.mark.parametrize("causal", [True, False])
def test_different_q_and_kv_packs(fw, lq, lk, causal):
    """Chunked-prefill shape (Lq < Lk), Lq > Lk (rows without visible keys when causal), empty KV."""
    run_case(fw, wl_prefill(causal=causal), lq, lk)


@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_256(fw, causal):
    run_case(fw, wl_prefill(hq=4, hkv=2, d=256, causal=causal), [129, 300, 1])


def test_many_units_balance_path(fw):
    """More units than CTAs: the snake schedule over the longest-first list."""
    wl = wl_prefill(hq=16, hkv=4)
    lens = [int(x) for x in np.random.default_rng(3).integers(1, 700, size=24)]
    total = sum(lens) * 16
    rows = np.random.default_rng(4).choice(total, size=min(total, 3000), replace=False)
    run_case(fw, wl, lens, rows=np.sort(rows))


def test_output_guard_and_lse_optional(fw):
    wl = wl_prefill(hq=4, hkv=2)
    inp = to_device(make_prefill_inputs(wl, "cpu", [150, 20]))
    big = torch.full((172, 4, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    out = big[1:171]
    fw.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"], True, wl.scale,
                      out=out, return_lse=False)
    torch.cuda.synchronize()
    assert torch.all(big[0] == 3.0) and torch.all(big[171] == 3.0)
    ref_o, _, ref_a = oracle.varlen_prefill(inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu(), inp["cu_seqlens_q"].cpu(),
                                            inp["cu_seqlens_k"].cpu(), True, wl.scale, with_absv=True)
    compare(out.reshape(-1, 128), None, ref_o, None, "guard", absv=ref_a)


def test_invalid_prefill_arguments(fw):
    wl = wl_prefill(hq=4, hkv=2)
    d = to_device(make_prefill_inputs(wl, "cpu", [10, 20]))
    before = fw.launch_count()
    with pytest.raises(fw.FwError):
        fw.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"][:2], d["cu_seqlens_k"], True, 0.1)
    with pytest.raises(fw.FwError):
        fw.varlen_prefill(d["q"][..., :64], d["k"][..., :64], d["v"][..., :64], d["cu_seqlens_q"],
                          d["cu_seqlens_k"], True, 0.1)
    with pytest.raises(fw.FwError):
        fw.varlen_prefill(d["q"][:, :3], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], True, 0.1)
    assert fw.launch_count() == before


@pytest.mark.parametrize("name", ["varlen_gqa_prefill", "dense_causal_mha_hd256"])
def test_full_size_workloads_sampled_rows(fw, name):
    """The benchmark workloads at full size; 512 sampled rows checked against the oracle."""
    wl = WORKLOADS[name]
    d = make_prefill_inputs(wl, "cuda")
    out, lse = fw.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal, wl.scale)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    total = d["q"].shape[0] * wl.num_q_heads
    rows = np.sort(np.random.default_rng(9).choice(total, size=512, replace=False))
    ref_o, ref_l, ref_a = oracle.varlen_prefill(d["q"].cpu(), d["k"].cpu(), d["v"].cpu(), d["cu_seqlens_q"].cpu(),
                                                d["cu_seqlens_k"].cpu(), wl.causal, wl.scale, rows=rows, with_absv=True)
    compare(out.reshape(-1, out.shape[-1])[rows], lse.reshape(-1)[rows], ref_o, ref_l, name, absv=ref_a)


def test_no_keys_at_all(fw):
    """Every KV length zero: all rows give zero output and -inf LSE."""
    run_case(fw, wl_prefill(hq=4, hkv=2), [5, 130], [0, 0])


@pytest.mark.parametrize("scale", [1.0, 2.0, 4.0, -0.2])
@pytest.mark.parametrize("d", [128, 256])
def test_scale_extremes_exercise_anchor_replay(fw, scale, d):
    """Large scales spread scores over ~100 log2 units, so later tiles outgrow the
    first tile's anchor and the running-sum check replays them (Flywheel appendix
    A); a negative scale exercises the sign-aware masking.  The device counter
    shows the replays ran: a float64 walk of the same check over these inputs
    replays 234-1117 (row, tile) steps at scales 2 and 4 (5 and 63 at scale 1,
    none at -0.2)."""
    wl = PrefillWorkload("s", num_seqs=0, num_q_heads=4, num_kv_heads=2, head_dim_qk=d, head_dim_v=d,
                         causal=True, scale=scale, value_seed=41)
    fw.read_counters()                                   # reset
    run_case(fw, wl, [300, 700, 129])
    replays = fw.read_counters()["prefill_replays"]
    if abs(scale) >= 2.0:
        assert replays > 0, "the static-anchor check never replayed a tile"


@pytest.mark.parametrize("pos", [10, 100])
@pytest.mark.parametrize("d", [128, 256])
def test_anchor_replay_in_either_half_of_a_tile(fw, pos, d):
    """One key of the second KV tile scores ~50 log2 units above everything else
    for every query row (a shared direction in Q and a large K entry), so every
    row's running-sum check fails on that tile, with the key in the first (pos
    10) or the second (pos 100) half of the tile's 128 keys.  At head dim 128
    the softmax hands P to the MMA in two halves of 64 keys, so a failure in the
    second half comes after the first half's PV went out with the old anchor and
    is repaired in O; both must match the oracle."""
    wl = wl_prefill(hq=4, hkv=2, d=d, causal=False, seed=43)
    inp = make_prefill_inputs(wl, "cpu", [256, 40])
    inp["q"][:, :, 0] = 2.0
    big = 128 + pos
    inp["k"][big] = 0.0
    inp["k"][big, :, 0] = 200.0 * math.sqrt(d / 128)   # the same score after the 1/sqrt(d) scale
    ref_o, ref_l, ref_a = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                                wl.causal, wl.scale, with_absv=True)
    dev = to_device(inp)
    fw.read_counters()                                   # reset
    out, lse = fw.varlen_prefill(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"], wl.causal,
                                 wl.scale)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert fw.read_counters()["prefill_replays"] >= 256 * 4, "every row of the first sequence replays once"
    compare(out.reshape(-1, out.shape[-1]), lse.reshape(-1), ref_o, ref_l, f"planted key at {pos}", absv=ref_a)


@pytest.fixture
def online(fw):
    """The prefill in its online-softmax mode (conditional rescale) for one test."""
    fw.set_option(fw.FW_OPT_PREFILL_SOFTMAX, 1)
    yield fw
    fw.set_option(fw.FW_OPT_PREFILL_SOFTMAX, 0)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_online_mode_ragged_batch(online, d, causal):
    """The conditional-rescale mode on ragged batches, empty and one-row sequences included."""
    run_case(online, wl_prefill(d=d, causal=causal), [130, 1, 257, 64, 0, 400])


@pytest.mark.parametrize("d", [128, 256])
def test_online_mode_different_packs(online, d):
    run_case(online, wl_prefill(d=d), [100, 5, 300, 7], [500, 5, 300, 0])


@pytest.mark.parametrize("scale", [2.0, -0.2])
@pytest.mark.parametrize("d", [128, 256])
def test_online_mode_rescales(online, scale, d):
    """Scores spread over ~100 log2 units: row maxima rise tile after tile, so the
    base moves often and l and O are rescaled in TMEM."""
    wl = PrefillWorkload("s", num_seqs=0, num_q_heads=4, num_kv_heads=2, head_dim_qk=d, head_dim_v=d,
                         causal=True, scale=scale, value_seed=41)
    run_case(online, wl, [300, 700, 129])


@pytest.mark.parametrize("name", ["varlen_gqa_prefill", "dense_causal_mha_hd256"])
def test_online_mode_full_size_sampled_rows(online, name):
    """Both softmax modes give the same result up to rounding at full size."""
    wl = WORKLOADS[name]
    d = make_prefill_inputs(wl, "cuda")
    out, lse = online.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal,
                                     wl.scale)
    torch.cuda.synchronize()
    assert online.device_status() == 0
    total = d["q"].shape[0] * wl.num_q_heads
    rows = np.sort(np.random.default_rng(10).choice(total, size=512, replace=False))
    ref_o, ref_l, ref_a = oracle.varlen_prefill(d["q"].cpu(), d["k"].cpu(), d["v"].cpu(), d["cu_seqlens_q"].cpu(),
                                                d["cu_seqlens_k"].cpu(), wl.causal, wl.scale, rows=rows, with_absv=True)
    compare(out.reshape(-1, out.shape[-1])[rows], lse.reshape(-1)[rows], ref_o, ref_l, name + " online", absv=ref_a)


@pytest.mark.parametrize("name", ["varlen_gqa_prefill", "dense_causal_mha_hd256"])
def test_repeated_launches_are_bitwise_identical(fw, name):
    """Every launch writes the same bytes: an accumulator read before its last
    MMA has landed, or a ring slot refilled while still in use, shows up as
    drift between launches.  Benchmark workloads at full size, four launches."""
    wl = WORKLOADS[name]
    d = make_prefill_inputs(wl, "cuda")
    args = (d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal, wl.scale)
    out0, lse0 = fw.varlen_prefill(*args)
    for _ in range(3):
        out, lse = fw.varlen_prefill(*args)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))
