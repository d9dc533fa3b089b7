"""fw_paged_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a runtime that owns the whole device pool and forbids
cudaMalloc in its execute step, a loop that cannot take an allocation's
implicit synchronisation) pass their own output buffers and get the scratch
from the library's fixed device array.  These tests call it through the C ABI
and require it to agree with fw_paged_decode, within the parity tolerance the
other GPU tests use, on two calls in a row (the second call reuses the scratch
the first one left behind).  This file is collected last so that a failure
here never hides the other tests.
"""
import math

import pytest
import torch

from ragged_softmax_attention_gb300.workloads import DecodeWorkload, make_decode_inputs
from tests.gpu_common import LSE_TOL, OUT_TOL, built_library

pytestmark = pytest.mark.gpu


def _inputs(batch, lens, q_len=1, hq=40, hkv=8, ps=128):
    wl = DecodeWorkload("noalloc", batch=batch, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim_qk=128, head_dim_v=128, page_size=ps, scale=1.0 / math.sqrt(128),
                        seq_lens=tuple(lens), value_seed=77, spare_pages=2)
    return make_decode_inputs(wl, "cuda")


def _close(a_out, a_lse, b_out, b_lse):
    ref = b_out.float()
    bound = OUT_TOL * torch.clamp(ref.abs(), min=1.0)
    assert torch.isfinite(a_out.float()).all()
    assert ((a_out.float() - ref).abs() <= bound).all()
    fin = torch.isfinite(b_lse)
    assert torch.equal(torch.isfinite(a_lse), fin)
    if fin.any():
        assert (a_lse[fin] - b_lse[fin]).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("lens,q_len,hq,hkv,ps", [
    ((9000, 130, 4100, 1, 2049, 700, 32768, 12), 1, 40, 8, 128),   # long rows split across CTAs
    ((37, 200, 0, 513), 3, 8, 2, 16),                               # small pages, causal rows, empty row
])
def test_noalloc_matches_allocating_decode_twice(lens, q_len, hq, hkv, ps):
    fw = built_library()
    d = _inputs(len(lens), lens, q_len, hq, hkv, ps)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    ref_out, ref_lse = fw.paged_decode(*args)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        fw.paged_decode_noalloc(*args, out=out, lse=lse)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        _close(out, lse, ref_out, ref_lse)


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
