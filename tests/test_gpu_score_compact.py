"""dspark_score_compact: steps a1-a4 in one launch.

"DFlash to DSpark in SGLang", sections "DSpark: a sequential head and a
verify budget", "Zero-overhead scheduling and kernels" (the verify-length
top-k) and "Ragged verify under full CUDA graphs" (the packing).

The fused call must write what dspark_score_budget followed by
dspark_compact writes, bit for bit, and its step must equal the oracle.
The shapes reach each way the finishing CTA can run: one request per thread
with everything in shared memory (conf loaded as float4 or one by one), the
general finish past 256 requests or when the packing inputs do not fit,
and the fixed budget's one-thread-per-slot kernel.
"""
import numpy as np
import pytest
import torch

from confidence_driven_speculative_gb300 import binding
from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import compare_with_oracle, gpu_step, to_device

pytestmark = pytest.mark.gpu

SCORE_OUT = ("conf", "survival", "L0", "L", "draft_off", "row_off", "packed_ids", "packed_pos",
             "row_req", "row_k")


def two_ways(inp_cpu):
    """The score and packing outputs of the two calls and of the fused one."""
    inp = to_device(inp_cpu)
    B, g, V, d = inp["B"], inp["gamma"], inp["V"], inp["d"]
    outs = []
    for fused in (False, True):
        bufs = binding.StepBuffers(B, g, V, d)
        for k in SCORE_OUT:   # stale values the calls must overwrite
            getattr(bufs, k).fill_(-5)
        bufs.bind(inp, seq_lens_commit=inp["seq_lens"].clone())
        if fused:
            binding.dspark_score_compact(bufs.step)
        else:
            binding.dspark_score_budget(bufs.step)
            binding.dspark_compact(bufs.step)
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        outs.append({k: getattr(bufs, k).cpu().numpy() for k in SCORE_OUT})
    return outs


CASES = [
    # (workload, B, gamma, d, cap_T, cost_c, fixed_budget)
    ("mixed", 1, 16, 7168, -1, 0.3, -1),      # B = 1
    ("mixed", 24, 8, 256, 60, 0.05, -1),      # cap binding, float4 conf loads
    ("mixed", 256, 16, 256, 768, 0.3, -1),    # the B = 256 shape, T = 768
    ("mixed", 256, 16, 64, 1000, 0.0, -1),    # every key a candidate
    ("tiny", 256, 15, 64, 900, 0.1, -1),      # gamma % 4 != 0: scalar conf loads, fp32 hidden
    ("mixed", 200, 7, 64, 10**6, 0.2, -1),    # a cap that does not bind
    ("mixed", 100, 9, 64, 0, 0.2, -1),        # T = 0
    ("mixed", 185, 64, 64, 3000, 0.0, -1),    # gamma = 64: the fused call's packing
                                              # inputs do not fit, so its finish is the
                                              # general one and the unfused call's the fast one
    ("mixed", 300, 4, 64, 500, 0.0, -1),      # past 256 requests: the general finish
    ("mixed", 600, 16, 64, 5000, 0.0, -1),    # curves re-read from memory
    ("mixed", 37, 7, 64, -1, 0.3, 3),         # fixed budgets
    ("mixed", 256, 16, 64, -1, 0.3, 16),
    ("mixed", 5, 4, 64, -1, 0.3, 0),
    ("mixed", 300, 4, 64, -1, 0.3, 9),
]


@pytest.mark.parametrize("case", CASES)
def test_fused_equals_the_two_calls(cuda_lib, case):
    wl, B, g, d, T, c, F = case
    base = W.TINY if wl == "tiny" else W.MIXED_B256
    inp = W.make_inputs(base, 30 + B, B=B, gamma=g, V=256, d=d, cap_T=T, cost_c=c,
                        fixed_budget=F)
    two, one = two_ways(inp)
    for k in SCORE_OUT:
        if F >= 0 and k in ("conf", "survival", "L0"):
            continue  # the fixed budget writes none of these
        assert np.array_equal(two[k], one[k]), k


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_fused_step_equals_the_oracle(cuda_lib, case, Tm):
    wl, B, g, d, T, c, F = case
    base = W.TINY if wl == "tiny" else W.MIXED_B256
    V = 20000 if B <= 64 else 520
    inp = W.make_inputs(base, 50 + B, B=B, gamma=g, V=V, d=d, cap_T=T, cost_c=c,
                        fixed_budget=F, temperature=Tm)
    gpu, _ = gpu_step(to_device(inp), fused=True)
    compare_with_oracle(W.to_numpy(inp), gpu)
    if T >= 0:
        assert gpu["L"].sum() <= T


def test_every_key_equal(cuda_lib):
    """A large head bias makes every confidence 1.0 in fp32, so every gain
    S_{b,k} is 1 and the cap keeps the first T keys in (b, k) order: the
    select's case where the largest and smallest key agree in every bit."""
    B, g, T = 24, 8, 50
    inp = W.make_inputs(W.MIXED_B256, 3, B=B, gamma=g, V=256, d=64, cap_T=T, cost_c=0.5)
    inp["head_bias"] = torch.full_like(inp["head_bias"], 200.0)
    two, one = two_ways(inp)
    want = np.zeros(B, np.int32)
    want[:T // g] = g
    want[T // g] = T % g
    for out in (two, one):
        assert np.all(out["survival"] == 1.0)
        assert np.all(out["L0"] == g)
        assert np.array_equal(out["L"], want)
    gpu, _ = gpu_step(to_device(inp), fused=True)
    compare_with_oracle(W.to_numpy(inp), gpu)


def test_two_key_values(cuda_lib):
    """Requests whose confidences are 1.0 or 0.5 exactly: the gains are
    powers of two, so many keys tie; ties go to the lower (b, k)."""
    B, g, T = 40, 6, 70
    inp = W.make_inputs(W.MIXED_B256, 4, B=B, gamma=g, V=256, d=64, cap_T=T, cost_c=0.01)
    # bias 200 gives conf 1.0; the hidden rows of odd requests are zero and
    # their bias 0 gives conf sigmoid(0) = 0.5
    bias = torch.full_like(inp["head_bias"], 200.0)
    bias[1::2] = 0.0
    inp["head_bias"] = bias
    inp["hidden"][1::2] = 0
    inp["sts_tau"] = torch.ones_like(inp["sts_tau"])
    two, one = two_ways(inp)
    # keys: even requests 1 (x g), odd requests 0.5, 0.25, ..., 0.5^g
    keys = []
    for b in range(B):
        for k in range(g):
            keys.append(((1.0 if b % 2 == 0 else 0.5 ** (k + 1)), b, k))
    keys.sort(key=lambda t: (-t[0], t[1], t[2]))
    want = np.zeros(B, np.int32)
    for _, b, _ in keys[:T]:
        want[b] += 1
    for out in (two, one):
        assert np.array_equal(out["L"], want)
    gpu, _ = gpu_step(to_device(inp), fused=True)
    compare_with_oracle(W.to_numpy(inp), gpu)


def test_packing_padding_and_nulls(cuda_lib):
    """Rows past N_rows carry the padding values; NULL last tokens and
    cached lengths pack as -1 and 0."""
    B, g = 10, 5
    inp = to_device(W.make_inputs(W.MIXED_B256, 8, B=B, gamma=g, V=256, d=64, cap_T=20,
                                  cost_c=0.2))
    bufs = binding.StepBuffers(B, g, 256, 64)
    bufs.bind(inp)
    bufs.step.last_tokens = None
    bufs.step.seq_lens_in = None
    binding.dspark_score_compact(bufs.step)
    torch.cuda.synchronize()
    n = int(bufs.row_off[B].item())
    L = bufs.L.cpu().numpy()
    ro = bufs.row_off.cpu().numpy()
    ids = bufs.packed_ids.cpu().numpy()
    pos = bufs.packed_pos.cpu().numpy()
    req = bufs.row_req.cpu().numpy()
    kk = bufs.row_k.cpu().numpy()
    drafts = inp["draft_tokens"].cpu().numpy()
    assert n == L.sum() + B
    for b in range(B):
        for j in range(L[b] + 1):
            r = ro[b] + j
            assert req[r] == b and kk[r] == j and pos[r] == j
            assert ids[r] == (-1 if j == 0 else drafts[b, j - 1])
    assert np.all(ids[n:] == -1) and np.all(pos[n:] == 0)
    assert np.all(req[n:] == -1) and np.all(kk[n:] == -1)
