"""Parity of the CUDA step (through the C ABI) with the CPU oracle.

Every integer output (L0, L, offsets, packed arrays, accept lengths, emitted
tokens, committed lengths) must match exactly, apart from decisions the oracle
flags as near ties; conf/survival within 1e-5 absolute; p(d), q(d) within
1e-3 relative.  Workloads: the five synthetic configurations at full size,
plus small shapes that span several vocab tiles with a ragged tail, and the
method's degenerate cases.
"""
import numpy as np
import pytest
import torch

from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import compare_with_oracle, gpu_step, outputs_of, to_device

pytestmark = pytest.mark.gpu


def run_and_compare(inp_cpu, fused=False, **kw):
    gpu, bufs = gpu_step(to_device(inp_cpu), fused=fused)
    stats = compare_with_oracle(W.to_numpy(inp_cpu), gpu, **kw)
    # the near-tie counts of every case (shown with pytest -s)
    print(f"parity {inp_cpu['workload']} B={inp_cpu['B']} V={inp_cpu['V']} "
          f"Tm={inp_cpu['temperature']}: {stats}")
    return gpu, stats, bufs


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_tiny_workload(cuda_lib, Tm):
    for step in range(3):
        run_and_compare(W.make_inputs(W.TINY, step, temperature=Tm))


@pytest.mark.parametrize("T", [0, 1, 3, 7, 24, -1])
@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_tiny_cap_binding(cuda_lib, T, Tm):
    inp = W.make_inputs(W.TINY, 5, temperature=Tm, cap_T=T, cost_c=0.05)
    gpu, _, _ = run_and_compare(inp)
    if T >= 0:
        assert gpu["L"].sum() <= T


@pytest.mark.parametrize("c", [-0.5, 0.0, 0.999, 1.0, 1.5])
def test_cost_edges(cuda_lib, c):
    inp = W.make_inputs(W.TINY, 1, cost_c=c, cap_T=-1)
    gpu, _, _ = run_and_compare(inp)
    if c <= 0:
        assert np.all(gpu["L"] == 8)
    if c >= 1.0:
        assert np.all(gpu["L"] == 0)


@pytest.mark.parametrize("F", [0, 3, 8, 20])
def test_fixed_budget(cuda_lib, F):
    inp = W.make_inputs(W.TINY, 2, cap_T=-1, fixed_budget=F)
    gpu, _, _ = run_and_compare(inp)
    assert np.all(gpu["L"] == min(F, 8))


# The cap's candidate sets on either side of the kernel's shared-memory
# limits.  Up to 256 requests one thread each holds a request's keys (the
# fast finish); past that the general finish lists up to 4096 keys and holds
# up to 8192 survival values on chip.
@pytest.mark.parametrize("B,T,c", [
    (256, 1000, 0.0),    # 4096 candidates, one request per thread
    (400, 2000, 0.0),    # 6400 candidates, curves on chip: the unlisted select
    (600, 5000, 0.0),    # 9600 candidates, curves re-read from memory
    (600, 700, 0.45),    # curves re-read from memory, fewer candidates
])
def test_cap_candidate_sets(cuda_lib, B, T, c):
    inp = W.make_inputs(W.MIXED_B256, 20, B=B, V=256, d=64, cap_T=T, cost_c=c)
    gpu, _, _ = run_and_compare(inp)
    assert gpu["L"].sum() <= T


# Small shapes: several vocab tiles (16 KB each) with a ragged tail, odd B and
# gamma, both dtypes, both modes.
SHAPES = [
    # (B, gamma, V, d, dtype)
    (1, 1, 8, 8, "bf16"),
    (3, 5, 8200, 40, "bf16"),      # 2 tiles, the second 16 bytes
    (37, 7, 20000, 264, "bf16"),   # 3 tiles, ragged
    (5, 16, 12292, 100, "f32"),    # 4 fp32 tiles, ragged
    (300, 4, 520, 64, "bf16"),     # many requests, one tile each
    (9, 64, 1000, 16, "bf16"),     # the largest gamma
    (12, 16, 70000, 64, "bf16"),   # the small-batch kernel: 9 slices of 8192 ids
    (16, 12, 40000, 32, "f32"),    # the small-batch kernel, fp32, its largest batch
    (17, 12, 40000, 32, "bf16"),   # one past it: the persistent kernel
    (8, 16, 151936, 64, "bf16"),   # small batch, rows of 19 tiles: rejections go to the tail kernel
    (6, 40, 40000, 16, "bf16"),    # the tail kernel with a long block (gamma = 40)
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("Tm", [0.0, 0.8])
def test_small_shapes(cuda_lib, shape, Tm):
    B, g, V, d, dt = shape
    base = W.TINY if dt == "f32" else W.MIXED_B256
    for step, (T, c) in enumerate([(-1, 0.3), (max(1, B * g // 3), 0.05)]):
        inp = W.make_inputs(base, 10 + step, B=B, gamma=g, V=V, d=d, temperature=Tm,
                            cap_T=T, cost_c=c)
        run_and_compare(inp)


def test_draft_equals_target_accepts_everything(cuda_lib):
    inp = W.make_inputs(W.MIXED_B256, 3, B=16, V=20000, d=64, cap_T=-1, cost_c=0.0)
    inp["draft_logits"] = inp["target_dense"][:, :-1].clone()
    gpu, _, _ = run_and_compare(inp)
    assert np.array_equal(gpu["accept_len"], gpu["L"])


@pytest.mark.parametrize("Tm", [0.0, 1.0])
@pytest.mark.parametrize("B,V", [(64, 20000), (12, 70000)])
def test_first_drafts_rejected(cuda_lib, Tm, B, V):
    """Drafts from an unrelated distribution: nearly every request rejects
    at its first draft, so most decisions take the residual path (sampling)
    or the argmax correction (greedy), and the bonus rows of those requests
    are not needed -- the verify may skip them.  At B = 12 with rows of nine
    tiles the small-batch verify lists nearly every request for its tail
    kernel."""
    inp = W.make_inputs(W.MIXED_B256, 7, B=B, V=V, d=64, cap_T=-1, cost_c=0.0,
                        temperature=Tm)
    g = torch.Generator().manual_seed(77)
    dl = torch.randn(inp["draft_logits"].shape, generator=g) * 4.0
    inp["draft_logits"] = dl.to(inp["draft_logits"].dtype)
    if Tm == 0.0:
        # greedy drafts that are never the target's argmax
        inp["draft_tokens"] = (inp["target_dense"][:, :-1].float().argmax(-1) + 1).to(torch.int32) % V
    else:
        gum = -torch.log(-torch.log(torch.rand(dl.shape, generator=g).clamp_min(1e-20)))
        inp["draft_tokens"] = (dl.float() + gum).argmax(-1).to(torch.int32)
    gpu, _, _ = run_and_compare(inp)
    assert np.all(gpu["L"] == 16)
    assert np.mean(gpu["accept_len"] == 0) > 0.8


def test_out_of_range_drafts_are_rejected(cuda_lib):
    for Tm in (0.0, 1.0):
        inp = W.make_inputs(W.MIXED_B256, 4, B=8, V=4096, d=64, cap_T=-1, cost_c=0.0,
                            temperature=Tm)
        inp["draft_tokens"][:, 2] = torch.tensor([-1, 4096, 10**6, -7, 4096, 5000, -2, 9999],
                                                 dtype=torch.int32)
        gpu, _, _ = run_and_compare(inp)
        assert np.all(gpu["accept_len"] <= 2)


def test_repeated_calls_reuse_the_workspace(cuda_lib):
    """Counters reset themselves: the same buffers give identical results on a
    second and third run, and the device status stays clean."""
    inp = to_device(W.make_inputs(W.MIXED_B256, 6, B=40, V=30000, d=128, cap_T=100))
    first, bufs = gpu_step(inp)
    for _ in range(2):
        again, _ = gpu_step(inp, bufs=bufs)
        for k in first:
            if first[k] is not None:
                assert np.array_equal(first[k], again[k]), k
    assert bufs.device_status() == 0


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_graph_replay_matches_direct_calls(cuda_lib, Tm):
    """The three calls captured as one CUDA graph (the compaction and the
    verify are programmatic dependents of the kernel before each) and replayed twice give the outputs of
    direct calls, bit for bit, on the same buffers, and each replay equals
    the oracle."""
    from confidence_driven_speculative_gb300 import binding
    inp_cpu = W.make_inputs(W.MIXED_B256, 9, B=24, V=20000, d=128, cap_T=60, temperature=Tm)
    inp = to_device(inp_cpu)
    ref, bufs = gpu_step(inp)  # direct calls; binds the ragged target rows
    names = ("L", "row_off", "packed_ids", "accept_len", "num_emitted", "out_tokens",
             "p_tok", "q_tok")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            binding.dspark_score_budget(bufs.step)
            binding.dspark_compact(bufs.step)
            binding.dspark_verify(bufs.step)
    torch.cuda.current_stream().wait_stream(side)
    commit = bufs._keep["seq_lens_commit"]
    for _ in range(2):
        for k in ("accept_len", "num_emitted", "out_tokens"):
            getattr(bufs, k).fill_(-7)
        commit.copy_(inp["seq_lens"])
        g.replay()
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        for k in names:
            assert np.array_equal(getattr(bufs, k).cpu().numpy(), ref[k]), k
        assert np.array_equal(commit.cpu().numpy(), ref["seq_lens_commit"])
        compare_with_oracle(W.to_numpy(inp_cpu), outputs_of(bufs, commit))


def _graph_over_totals(workload, steps, B, V, d, min_totals, temperature=1.0, fused=False):
    """One capture of the step -- score, compact (or the fused
    dspark_score_compact), a fixed-shape target stand-in over the batch's
    capacity of rows, verify -- replayed on input sets whose packed totals
    differ.  Each replay equals direct calls on that set and the oracle.
    Returns the packed totals seen."""
    from confidence_driven_speculative_gb300 import binding
    sets_cpu = [W.make_inputs(workload, s, B=B, V=V, d=d, cap_T=-1, temperature=temperature)
                for s in steps]
    for st in sets_cpu:
        st["seed"] = 5                      # a host scalar fixed at capture
    sets = [to_device(st) for st in sets_cpu]
    keys = ("hidden", "head_w", "head_bias", "sts_tau", "draft_tokens", "draft_logits",
            "target_dense", "last_tokens", "seq_lens")
    live = {k: (v.clone() if k in keys else v) for k, v in sets[0].items()}
    g1 = live["gamma"] + 1
    bufs = binding.StepBuffers(B, live["gamma"], V, d)
    commit = live["seq_lens"].clone()
    bufs.bind(live, seq_lens_commit=commit)
    tgt = torch.empty((B * g1, V), dtype=live["target_dense"].dtype, device="cuda")
    bufs.bind_target(tgt)
    flat = live["target_dense"].view(B * g1, V)

    def step():
        if fused:
            binding.dspark_score_compact(bufs.step)
        else:
            binding.dspark_score_budget(bufs.step)
            binding.dspark_compact(bufs.step)
        idx = (bufs.row_req.clamp(min=0) * g1 + bufs.row_k.clamp(min=0)).long()
        torch.index_select(flat, 0, idx, out=tgt)
        binding.dspark_verify(bufs.step)

    step()                                  # warm-up outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    totals = []
    for st, st_cpu in zip(sets, sets_cpu):
        ref, _ = gpu_step(st)
        for k in keys:
            live[k].copy_(st[k])
        commit.copy_(st["seq_lens"])
        for k in ("accept_len", "num_emitted", "out_tokens"):
            getattr(bufs, k).fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        n = int(ref["draft_off"][B])
        for k in ("L", "row_off", "packed_ids", "accept_len", "num_emitted", "out_tokens"):
            assert np.array_equal(getattr(bufs, k).cpu().numpy(), ref[k]), k
        for k in ("p_tok", "q_tok"):
            assert np.array_equal(getattr(bufs, k).cpu().numpy()[:n], ref[k][:n]), k
        assert np.array_equal(commit.cpu().numpy(), ref["seq_lens_commit"])
        compare_with_oracle(W.to_numpy(st_cpu), outputs_of(bufs, commit))
        totals.append(int(ref["row_off"][B]))
    assert len(set(totals)) >= min_totals, totals
    return totals


def test_one_graph_serves_every_packed_total(cuda_lib):
    """Four batches of B=24 through one captured graph, at least three
    distinct packed totals: the kernels take the total from device memory, so
    no per-total graph tier is needed."""
    _graph_over_totals(W.MIXED_B256, range(40, 44), 24, 20000, 128, min_totals=3)


def test_one_graph_of_the_fused_call_serves_every_packed_total(cuda_lib):
    """As above with dspark_score_compact captured in place of the first
    two calls (the verify then depends on the score kernel directly)."""
    _graph_over_totals(W.MIXED_B256, range(40, 44), 24, 20000, 128, min_totals=3, fused=True)


def test_one_graph_serves_the_b1_latency_shape(cuda_lib):
    """The B=1 latency shape (V = 129280, d = 7168) through one captured
    graph over several steps (its own greedy verify, then sampling), each
    replay checked against the oracle."""
    w = W.LATENCY_B1
    for Tm in (None, 1.0):
        for fused in (False, True):
            _graph_over_totals(w, range(5), 1, w.V, w.d, min_totals=1, temperature=Tm,
                               fused=fused)


def test_empty_batch(cuda_lib):
    from confidence_driven_speculative_gb300 import binding
    step = binding.DsparkStep()
    step.B, step.gamma, step.V, step.d = 0, 4, 16, 8
    for fn in (binding.dspark_score_budget, binding.dspark_score_compact, binding.dspark_compact,
               binding.dspark_verify):
        assert fn(step) == binding.DSPARK_OK


def test_qwen3_8b_shape(cuda_lib):
    for step in range(2):
        run_and_compare(W.make_inputs(W.QWEN3_8B, step), fused=step == 1)


def test_latency_b1(cuda_lib):
    for step in range(3):
        run_and_compare(W.make_inputs(W.LATENCY_B1, step), fused=step > 0)


@pytest.mark.slow
def test_mixed_b256_dynamic(cuda_lib):
    for step in range(2):
        _, stats, _ = run_and_compare(W.make_inputs(W.MIXED_B256, step), fused=step == 1)


@pytest.mark.slow
def test_mixed_b256_fixed_budget(cuda_lib):
    gpu, _, _ = run_and_compare(W.make_inputs(W.MIXED_B256, 0, cap_T=-1, fixed_budget=5))
    assert np.all(gpu["L"] == 5)


@pytest.mark.slow
def test_qwen3_14b_sweep(cuda_lib):
    for step in range(2):
        run_and_compare(W.make_inputs(W.QWEN3_14B_SWEEP, step))
