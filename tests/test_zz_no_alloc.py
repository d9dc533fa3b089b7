"""fw_paged_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a runtime that owns the whole device pool and forbids
cudaMalloc in its execute step, a loop that cannot take an allocation's
implicit synchronisation) pass their own output buffers and get the scratch
from the library's fixed device array.  These tests call it through the C ABI
on two calls in a row (the second call reuses the scratch the first one left
behind) and require each result to match the fp64 oracle within the parity
bar every other GPU test uses, and to agree with fw_paged_decode on the same
inputs.  The cases cover every decode kernel family that can use the fixed
array: grouped-query heads (hd 128) with long rows split across CTAs, small
pages with causal multi-token rows and an empty row, and latent heads
(Dk 576 / Dv 512, 512-float partial rows) with forced splits.  This file is
collected last so that a failure here never hides the other tests.
"""
import math

import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import DecodeWorkload, make_decode_inputs
from tests.gpu_common import LSE_TOL, OUT_TOL, built_library, compare

pytestmark = pytest.mark.gpu


def _workload(lens, q_len, hq, hkv, ps, latent):
    if latent:
        return DecodeWorkload("noalloc-latent", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                              head_dim_qk=576, head_dim_v=512, page_size=ps, scale=0.07216882,
                              seq_lens=tuple(lens), latent=True, value_seed=79, spare_pages=2)
    return DecodeWorkload("noalloc", batch=len(lens), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim_qk=128, head_dim_v=128, page_size=ps, scale=1.0 / math.sqrt(128),
                          seq_lens=tuple(lens), value_seed=77, spare_pages=2)


def _agree(a_out, a_lse, b_out, b_lse):
    """Two GPU results within the absolute parity bar of each other."""
    assert torch.isfinite(a_out.float()).all()
    assert (a_out.float() - b_out.float()).abs().max().item() <= OUT_TOL
    fin = torch.isfinite(b_lse)
    assert torch.equal(torch.isfinite(a_lse), fin)
    if fin.any():
        assert (a_lse[fin] - b_lse[fin]).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("lens,q_len,hq,hkv,ps,latent,chunk", [
    ((9000, 130, 4100, 1, 2049, 700, 32768, 12), 1, 40, 8, 128, False, 0),   # long rows split across CTAs
    ((37, 200, 0, 513), 3, 8, 2, 16, False, 0),                               # small pages, causal rows, empty row
    ((3000, 1100), 4, 128, 1, 64, True, 512),                                 # latent heads, forced splits
])
def test_noalloc_matches_oracle_twice(lens, q_len, hq, hkv, ps, latent, chunk):
    fw = built_library()
    wl = _workload(lens, q_len, hq, hkv, ps, latent)
    inp = make_decode_inputs(wl, "cpu")
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], with_absv=True)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if latent:
        d["v_cache"] = d["k_cache"][..., :512]          # values: the first 512 columns of the latent row
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, chunk)
    try:
        alloc_out, alloc_lse = fw.paged_decode(*args)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        for call in range(2):
            out = torch.full_like(alloc_out, float("nan"))
            lse = torch.full_like(alloc_lse, float("nan"))
            fw.paged_decode_noalloc(*args, out=out, lse=lse)
            torch.cuda.synchronize()
            assert fw.device_status() == 0
            compare(out, lse, ref_o, ref_l, what=f"noalloc call {call} {wl.name} {lens}", absv=ref_a)
            _agree(out, lse, alloc_out, alloc_lse)
    finally:
        fw.set_option(fw.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def test_noalloc_rejects_scratch_beyond_its_limit():
    """Shapes whose scratch exceeds the fixed 64 MiB return FW_ERR_WORKSPACE and launch nothing."""
    fw = built_library()
    q = torch.zeros(64, 1, 40, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(4, 128, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(64, 4096, dtype=torch.int32, device="cuda")      # bound: 4096 pages x 128 keys per row
    sl = torch.ones(64, dtype=torch.int32, device="cuda")
    out = torch.empty(64, 1, 40, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, 1, 40, dtype=torch.float32, device="cuda")
    plan = fw.plan_decode(64, 1, 40, 8, 128, 4096 * 128)
    assert plan["workspace_bytes"] > 64 << 20
    before = fw.launch_count()
    with pytest.raises(fw.FwError) as e:
        fw.paged_decode_noalloc(q, cache, cache, bt, sl, 0.1, out=out, lse=lse)
    assert e.value.status == 3 and "fixed scratch" in str(e.value)
    assert fw.launch_count() == before
