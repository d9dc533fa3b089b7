"""The bounded device waits: a wait that runs out reports FW_ERR_DEVICE_TIMEOUT
instead of trapping, and the library stays usable.

"Flywheel Attention", section 3.1: a failed check raises a flag the host
reads instead of faulting.  The kernels' mbarrier waits follow that rule:
after FW_OPT_WAIT_TIMEOUT_MS a wait gives up, records FW_ERR_DEVICE_TIMEOUT in
the device status word, raises the CTA's abort flag so every other wait
returns at once, and the CTA leaves once the copies and MMAs it issued have
landed.  The test hook FW_OPT_TEST_STALL makes the grouped-query decode's copy
warp wait, before it copies anything, on a barrier that nothing completes:
the wait runs out with no copy or MMA in flight, so the failure path runs
without risk to the device.  The CTA-pair kernels are not used here.
"""
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs
from tests.gpu_common import built_library, compare, to_device

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_next_call_is_correct():
    fw = built_library()
    wl = WORKLOADS["tiny_paged_decode"]
    inp = make_decode_inputs(wl, "cpu")
    d = to_device(inp)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    assert fw.device_status() == 0
    fw.set_option(fw.FW_OPT_WAIT_TIMEOUT_MS, 1)            # the shortest limit
    fw.set_option(fw.FW_OPT_TEST_STALL, 1)
    try:
        fw.paged_decode(*args)                             # the call itself is accepted
        torch.cuda.synchronize()
        assert fw.device_status() == fw.FW_ERR_DEVICE_TIMEOUT
    finally:
        fw.set_option(fw.FW_OPT_TEST_STALL, 0)
        fw.set_option(fw.FW_OPT_WAIT_TIMEOUT_MS, 2000)
    assert fw.device_status() == 0                         # reading the word cleared it
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                              inp["seq_lens"], inp["scale"], with_absv=True)
    for _ in range(2):
        out, lse = fw.paged_decode(*args)
        torch.cuda.synchronize()
        assert fw.device_status() == 0
        compare(out, lse, ref_o, ref_l, what="after a timed-out call", absv=ref_a)
