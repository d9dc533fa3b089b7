"""Non-causal paged decode on the GPU (fw_paged_decode_masked), through the C
ABI, against the fp64 oracle ("TokenSpeed-MLA 2.0.1", MLA decode:
causal_mask supports causal and non-causal execution; window_left starts row
i's history at max(0, K - q_len - window_left + i) either way).

Every query token of a row sees all n keys.  Covers the grouped-query BF16
and FP8 kernels, the latent kernels on CTA pairs, on one CTA and with packed
(token, head) rows, rows shorter than q_len, split-KV pieces, and (latent
layout) non-causal sliding windows with evicted pages; causal=True through
the same entry point matches fw_paged_decode bit for bit.
"""
import math

import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import DecodeWorkload, make_decode_inputs
from tests.gpu_common import BF16_UNIT, FP16_UNIT, built_library, compare, to_device
from tests.test_decode_window_gpu import evict_before_window

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    yield lib
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def wl_of(lens, q_len, hq, hkv, d=128, dv=None, ps=16, fp8=False, latent=False, seed=71):
    dv = dv or d
    scale = 0.07216882 if latent else 1.0 / math.sqrt(d)
    return DecodeWorkload("nc", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=d,
                          head_dim_v=dv, page_size=ps, scale=scale, seq_lens=tuple(lens), kv_fp8=fp8,
                          latent=latent, value_seed=seed, spare_pages=3)


def run_case(fw, wl, causal=False, window=-1, chunk=0):
    inp = make_decode_inputs(wl, "cpu")
    if window >= 0:
        inp = evict_before_window(inp, wl, window)
    ks, vs = (inp["k_scale"], inp["v_scale"]) if wl.kv_fp8 else (1.0, 1.0)
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], k_scale=ks, v_scale=vs,
                                              window_left=window, causal=causal, with_absv=True)
    d = to_device(inp)
    if wl.latent:
        d["v_cache"] = d["k_cache"][..., :wl.head_dim_v]
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        out, lse = fw.paged_decode_masked(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                          d["scale"], causal=causal, window_left=window, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    assert fw.device_status() == 0
    compare(out, lse, ref_o, ref_l, what=f"non-causal={not causal} window={window} {wl.seq_lens} q_len={wl.q_len}", absv=ref_a,
            p_unit=FP16_UNIT if wl.kv_fp8 else BF16_UNIT)
    return d, out, lse


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("q_len", [2, 4])
def test_grouped_query_noncausal(fw, fp8, q_len):
    """40/8 heads (G = 5 folded with the tokens), rows of 1..700 keys, some shorter than q_len."""
    run_case(fw, wl_of([1, 3, 130, 700], q_len, 40, 8, fp8=fp8))


def test_grouped_query_noncausal_hd256_and_splits(fw):
    run_case(fw, wl_of([2000, 5, 900], 3, 16, 2, d=256, ps=32), chunk=512)


@pytest.mark.parametrize("hq,hkv,q_len", [(128, 1, 4), (128, 2, 2), (96, 1, 4), (16, 1, 4)])
def test_latent_noncausal(fw, hq, hkv, q_len):
    """CTA pairs, one CTA, packed rows (H96, H16)."""
    run_case(fw, wl_of([1, 4, 300, 1100], q_len, hq, hkv, d=576, dv=512, ps=64, latent=True))


@pytest.mark.parametrize("window", [0, 50, 300])
def test_latent_noncausal_window(fw, window):
    """Non-causal with a window: each token's range starts at its own position
    minus W and runs to the row's end; pages before it are evicted."""
    run_case(fw, wl_of([3, 200, 1500], 4, 96, 1, d=576, dv=512, ps=32, latent=True), window=window)


def test_causal_through_masked_equals_paged_decode(fw):
    wl = wl_of([77, 500], 3, 40, 8)
    d, out, lse = run_case(fw, wl, causal=True)
    o2, l2 = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), l2.view(torch.int32))


def test_grouped_query_noncausal_window_is_rejected(fw):
    wl = wl_of([100], 2, 8, 2)
    d = to_device(make_decode_inputs(wl, "cpu"))
    before = fw.launch_count()
    with pytest.raises(fw.FwError):
        fw.paged_decode_masked(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"],
                               causal=False, window_left=10)
    assert fw.launch_count() == before
