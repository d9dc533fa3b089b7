"""The schedulers under a tight CTA cap (FW_OPT_MAX_CTAS), on the GPU, against
the fp64 oracle.

With a handful of persistent CTAs every CTA runs many units: the hd-128
prefill's four-slot unit queue wraps round many times and its counter hands
out every list entry, the hd-256 CTA pair walks the whole list alone, and the
decode ranges (tiles plus the empty slots that stand for piece starts) are
long and cross many unit boundaries, each a piece with its own partials.
With 4 CTAs and 2 KV heads the heads ride on the CTA index: two CTA pairs,
each pair walking the same ranges for the two heads.
"""
import math

import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import DecodeWorkload, PrefillWorkload, make_decode_inputs, \
    make_prefill_inputs
from tests.gpu_common import BF16_UNIT, FP16_UNIT, built_library, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    yield lib
    lib.set_option(lib.FW_OPT_MAX_CTAS, 0)


def capped(fw, ctas, call):
    fw.set_option(fw.FW_OPT_MAX_CTAS, ctas)
    try:
        result = call()
        torch.cuda.synchronize()
    finally:
        fw.set_option(fw.FW_OPT_MAX_CTAS, 0)
    assert fw.device_status() == 0
    return result


@pytest.mark.parametrize("d,ctas", [(128, 1), (128, 3), (256, 2), (256, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_with_few_ctas(fw, d, ctas, causal):
    wl = PrefillWorkload("few", num_seqs=0, num_q_heads=8, num_kv_heads=2, head_dim_qk=d, head_dim_v=d,
                         causal=causal, scale=1.0 / math.sqrt(d), value_seed=61)
    lens = [300, 1, 129, 700, 0, 256, 45]
    inp = make_prefill_inputs(wl, "cpu", lens)
    ref_o, ref_l, ref_a = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                                inp["cu_seqlens_k"], wl.causal, wl.scale, with_absv=True)
    dev = to_device(inp)
    out, lse = capped(fw, ctas, lambda: fw.varlen_prefill(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                                                          dev["cu_seqlens_k"], wl.causal, wl.scale))
    compare(out.reshape(-1, out.shape[-1]), lse.reshape(-1), ref_o, ref_l, f"prefill d={d} ctas={ctas}",
            absv=ref_a)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("ctas", [1, 3, 4])
def test_decode_with_few_ctas(fw, fp8, ctas):
    lens = (37, 1, 900, 129, 0, 300, 2000, 5)
    wl = DecodeWorkload("few", batch=len(lens), q_len=1, num_q_heads=8, num_kv_heads=2, head_dim_qk=128,
                        head_dim_v=128, page_size=32, scale=1.0 / math.sqrt(128), seq_lens=lens, kv_fp8=fp8,
                        value_seed=62, spare_pages=3)
    inp = make_decode_inputs(wl, "cpu")
    extra = {"k_scale": inp["k_scale"], "v_scale": inp["v_scale"]} if fp8 else {}
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], with_absv=True, **extra)
    d = to_device(inp)
    if fp8:
        call = lambda: fw.paged_decode_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                           d["scale"], inp["k_scale"], inp["v_scale"])
    else:
        call = lambda: fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                       d["scale"])
    out, lse = capped(fw, ctas, call)
    compare(out, lse, ref_o, ref_l, f"decode fp8={fp8} ctas={ctas}", absv=ref_a,
            p_unit=FP16_UNIT if fp8 else BF16_UNIT)
