"""A bounded device wait that runs out.

Every wait in the score and verify kernels gives up after the bound that
dspark_set_wait_timeout_ns sets (2 s by default), writes a status bit to the
workspace and returns; it never spins without a limit.  Here the bound is cut
to 100 ns for one verify launch, so the first waits for a copy or a queue
entry give up: the launch must still return, report the status, and after
dspark_workspace_init and the default bound restored, the next step must be
clean and equal to the oracle.
"""
import numpy as np
import pytest
import torch

from confidence_driven_speculative_gb300 import binding
from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import compare_with_oracle, gpu_step, to_device

pytestmark = pytest.mark.gpu

STATUS_WAIT = 1   # a wait on the shared-memory copy ring gave up
STATUS_QUEUE = 2  # a wait on other warps or CTAs gave up


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_short_wait_bound_gives_up_and_workspace_recovers(cuda_lib, Tm):
    # B = 96: the persistent verify kernel, whose producers, consumers and
    # deciders wait on one another (the small-batch kernel has no waits)
    inp_cpu = W.make_inputs(W.MIXED_B256, 12, B=96, V=20000, d=128, cap_T=-1, temperature=Tm)
    inp = to_device(inp_cpu)
    _, bufs = gpu_step(inp)  # a clean step binds every buffer
    default = binding.dspark_wait_timeout_ns()
    assert default == 2_000_000_000
    try:
        binding.dspark_set_wait_timeout_ns(100)
        assert binding.dspark_wait_timeout_ns() == 100
        binding.dspark_verify(bufs.step)
        torch.cuda.synchronize()  # the launch returned
        status = bufs.device_status()
    finally:
        binding.dspark_set_wait_timeout_ns(0)  # 0 restores the default
    assert binding.dspark_wait_timeout_ns() == default
    assert status & (STATUS_WAIT | STATUS_QUEUE), status
    assert status & ~(STATUS_WAIT | STATUS_QUEUE) == 0, status
    # The workspace is reset and the next step is clean and exact.
    binding.dspark_workspace_init(bufs.workspace.data_ptr(), bufs.ws_bytes)
    assert bufs.device_status() == 0
    gpu, _ = gpu_step(inp, bufs=bufs)
    compare_with_oracle(W.to_numpy(inp_cpu), gpu)
    assert np.all(gpu["num_emitted"] == gpu["accept_len"] + 1)
