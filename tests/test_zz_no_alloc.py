"""dspark_verify_noalloc -- the verify step on the library's fixed device
scratch, for callers that cannot allocate a workspace -- against
dspark_verify with a workspace.  Two calls in a row must give the workspace
path's outputs bit for bit (the same kernel runs on the same inputs) with a
clean device status.  The file sorts last, so it runs after every other test;
it also passes on its own, because the first call zeroes the scratch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from confidence_driven_speculative_gb300 import binding
from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import gpu_step, to_device

pytestmark = pytest.mark.gpu

VERIFY_OUTPUTS = ("accept_len", "num_emitted", "out_tokens", "p_tok", "q_tok")


def _run_noalloc(bufs, inp, status):
    """Scribble over what the verify step writes, restore the committed
    lengths, run the no-alloc entry point and return its outputs and device
    status.  p(d_k), q(d_k) are packed at draft_off[b] + k for the verified
    drafts (k < L_b), so only the first sum(L) entries are scribbled; the
    rest must stay as they were."""
    for k in ("accept_len", "num_emitted", "out_tokens"):
        getattr(bufs, k).fill_(-7)
    n_drafts = int(bufs.draft_off[bufs.B].item())
    for k in ("p_tok", "q_tok"):
        getattr(bufs, k)[:n_drafts] = float("nan")
    commit = bufs._keep["seq_lens_commit"]
    commit.copy_(inp["seq_lens"])
    status.fill_(-1)
    binding.dspark_verify_noalloc(bufs.step, status_out=status)
    torch.cuda.synchronize()
    out = {k: getattr(bufs, k).cpu().numpy() for k in VERIFY_OUTPUTS}
    out["seq_lens_commit"] = commit.cpu().numpy()
    return out, int(status.item())


def _inputs(case):
    if case == "tiny_sampling":
        return W.make_inputs(W.TINY, 0, temperature=1.0)
    if case == "tiny_greedy":
        return W.make_inputs(W.TINY, 1, temperature=0.0)
    if case == "ragged_sampling":
        return W.make_inputs(W.MIXED_B256, 6, B=40, V=30000, d=128, cap_T=100)
    return W.make_inputs(W.MIXED_B256, 0)  # B=256, gamma=16, V=129280


@pytest.mark.parametrize("case", ["tiny_sampling", "tiny_greedy", "ragged_sampling", "mixed_b256"])
def test_noalloc_matches_workspace_path_twice(cuda_lib, case):
    inp = to_device(_inputs(case))
    ref, bufs = gpu_step(inp)  # score, compact, verify with a workspace
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got, st = _run_noalloc(bufs, inp, status)
        assert st == 0
        for k in VERIFY_OUTPUTS + ("seq_lens_commit",):
            assert np.array_equal(ref[k], got[k], equal_nan=True), k


def test_noalloc_rejects_a_shape_beyond_its_scratch(cuda_lib):
    """B=1024, gamma=16, V=151936 needs more than the fixed scratch: refused
    before anything is enqueued, and an in-range call afterwards still
    matches the workspace path."""
    assert binding.dspark_workspace_size(1024, 16, 151936, 4096) > binding.DSPARK_NOALLOC_SCRATCH_BYTES
    step = binding.DsparkStep()
    step.B, step.gamma, step.V, step.d = 1024, 16, 151936, 4096
    assert binding.dspark_verify_noalloc(step, check=False) == binding.DSPARK_EWORKSPACE
    assert "static scratch" in binding.last_error()
    inp = to_device(_inputs("tiny_sampling"))
    ref, bufs = gpu_step(inp)
    got, st = _run_noalloc(bufs, inp, torch.empty(1, dtype=torch.int32, device="cuda"))
    assert st == 0
    for k in VERIFY_OUTPUTS:
        assert np.array_equal(ref[k], got[k], equal_nan=True), k


def test_graph_replay_after_a_call_of_another_shape(cuda_lib):
    """Capture a no-alloc verify of shape A, make an eager call of shape B
    (which re-zeroes the scratch for B's layout), then replay A's graph: the
    shape check runs on the device in stream order, so the replay zeroes for
    A again and equals dspark_verify with a workspace."""
    inp_a = to_device(_inputs("ragged_sampling"))
    ref_a, bufs_a = gpu_step(inp_a)
    inp_b = to_device(_inputs("tiny_sampling"))
    ref_b, bufs_b = gpu_step(inp_b)
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    got, st = _run_noalloc(bufs_a, inp_a, status)  # eager A, before any capture
    assert st == 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            binding.dspark_verify_noalloc(bufs_a.step, status_out=status)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        got_b, st_b = _run_noalloc(bufs_b, inp_b, status)  # eager B
        assert st_b == 0
        for k in VERIFY_OUTPUTS:
            assert np.array_equal(ref_b[k], got_b[k], equal_nan=True), k
        for k in ("accept_len", "num_emitted", "out_tokens"):
            getattr(bufs_a, k).fill_(-7)
        commit = bufs_a._keep["seq_lens_commit"]
        commit.copy_(inp_a["seq_lens"])
        status.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for k in VERIFY_OUTPUTS:
            assert np.array_equal(ref_a[k], getattr(bufs_a, k).cpu().numpy(), equal_nan=True), k
        assert np.array_equal(ref_a["seq_lens_commit"], commit.cpu().numpy())


@pytest.mark.slow
def test_noalloc_accepts_the_largest_documented_shape(cuda_lib):
    """B=512, gamma=16, V=151936 (the header's stated limit) is accepted and
    its device status is clean."""
    w = W.QWEN3_8B
    inp = to_device(W.make_inputs(w, 0, B=512, d=256, cap_T=-1))
    ref, bufs = gpu_step(inp)
    got, st = _run_noalloc(bufs, inp, torch.empty(1, dtype=torch.int32, device="cuda"))
    assert st == 0
    for k in VERIFY_OUTPUTS:
        assert np.array_equal(ref[k], got[k], equal_nan=True), k
