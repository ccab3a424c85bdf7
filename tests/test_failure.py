"""Failure detection without a GPU fault: a device wait that nothing ends
runs out its (short) limit, the kernel reports KDA_DEVICE_TIMEOUT in the
workspace status word, the host reads it, and the context stays usable for
a normal forward afterwards."""
import pytest
import torch

import kda_inputs as ki
from kda_testlib import assert_parity, run_gpu, run_oracle

KDA_DEVICE_TIMEOUT = 0x1


def test_selftest_rejects_bad_arguments():
    import gated_delta_rule_21_gb300 as kda
    L = kda.lib()
    assert L.kda_selftest_wait_timeout(None, 1000, None) == 1        # NULL workspace
    ws = torch.zeros(256, dtype=torch.uint8)
    assert L.kda_selftest_wait_timeout(ws.data_ptr(), 0, None) == 1   # limit < 1
    assert L.kda_selftest_wait_timeout(ws.data_ptr(), 1 << 40, None) == 1


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives():
    import gated_delta_rule_21_gb300 as kda
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    assert kda.read_device_status(ws) == 0
    kda.selftest_wait_timeout(ws, limit_cycles=1 << 20)   # ~0.5 ms of SM clock
    bits = kda.read_device_status(ws)
    assert bits & KDA_DEVICE_TIMEOUT
    kda.clear_device_status(ws)
    assert kda.read_device_status(ws) == 0
    # the context is still usable: a forward afterwards matches the oracle
    w = ki.WORKLOADS["fixed_bf16_h8_t1024"]
    x = ki.make_inputs(w, seed=5)
    o, fs = run_gpu(x)
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "forward after timeout o")
    assert_parity(fs, fs_ref, True, "forward after timeout final_state")
