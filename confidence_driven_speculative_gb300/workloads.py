"""Seeded synthetic inputs for the verify step.

This module only draws random inputs; it holds none of the step's arithmetic
(no confidence head, survival, cap, packing, softmax or accept rule).  The
same generated tensors feed both the CUDA library and the CPU oracle.

The pages measure on real models and datasets (gsm8k, arena-hard, poetry,
HumanEval; Qwen3 and DeepSeek-V4 targets).  None of them is available here, so
every workload is synthetic, with the shapes the pages name (Qwen3 vocabulary
151936; DeepSeek-class vocabulary 129280 and hidden size 7168) and value
distributions that mimic peaked ("code-like") and flat ("prose-like") targets
and drafts whose quality decays with block position (suffix decay, "DFlash to
DSpark in SGLang", section "DSpark: a sequential head and a verify budget").

Recipe shared by all workloads (per request b, draft position i = 0..gamma-1):

* hidden h[b,i,:] ~ N(0, 1); head weight w ~ N(0, 1/d); per-request bias;
  STS temperatures tau_i as listed.
* target logits z_p[b,j,:] for the gamma+1 ragged rows j = 0..gamma: a
  Gaussian background plus, for peaked workloads, a spike added at one
  uniformly drawn token index per row.
* draft logits z_q[b,i,:] = z_p[b,i,:] + N(0, sigma_i^2) with sigma_i growing
  in i (computed in fp32 before the single rounding to the storage dtype).
* drafted tokens: drawn from softmax(z_q / Tm) by the Gumbel-max trick when
  the workload samples (Tm > 0), or argmax z_q for a greedy drafter (Tm = 0);
  the tiny workload always draws at temperature 1 as its description says.
* last (root) tokens uniform in [0, V); cached lengths uniform in [16, 4096).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    d: int
    dtype: str              # "f32" or "bf16" (logits and hidden states)
    temperature: float      # 0 = greedy verify
    cost_c: float           # fixed c (ignored when c_range is set)
    cap_T: int              # < 0: no cap
    index: int              # seed namespace
    c_range: Optional[tuple] = None   # per-step c ~ U[lo, hi]
    draft_temperature: Optional[float] = None  # temperature of the drafter's draw
    description: str = ""


# The five workloads; the names say what they are.
TINY = Workload(
    "tiny_B4_g8_V1024_d256_fp32", B=4, gamma=8, V=1024, d=256, dtype="f32",
    temperature=1.0, cost_c=0.3, cap_T=24, index=1, draft_temperature=1.0,
    description="oracle-sized step: fp32, N(0,2^2) targets, draft noise 0.2+0.1i, "
                "bias 1, tau_i = 1+0.05i, c=0.3, T=24; greedy and Tm=1 runs")
QWEN3_8B = Workload(
    "qwen3_8b_shape_B32_g16_V151936_d4096_bf16", B=32, gamma=16, V=151936, d=4096,
    dtype="bf16", temperature=1.0, cost_c=0.25, cap_T=-1, index=2,
    description="N(0,3^2) + 8 spike targets, draft noise 0.3+0.08i, tau_i = 1+0.03i, "
                "c=0.25, no cap, Tm=1")
LATENCY_B1 = Workload(
    "latency_B1_g16_V129280_d7168_bf16", B=1, gamma=16, V=129280, d=7168, dtype="bf16",
    temperature=0.0, cost_c=0.15, cap_T=-1, index=3,
    description="N(0,2^2) + 10 spike target, draft noise 0.1+0.05i, c=0.15, greedy")
MIXED_B256 = Workload(
    "mixed_B256_g16_V129280_d7168_bf16", B=256, gamma=16, V=129280, d=7168,
    dtype="bf16", temperature=1.0, cost_c=0.35, cap_T=768, index=4,
    description="half code-like (N(0,2^2)+10 spike, noise 0.1+0.04i, bias +2), half "
                "prose-like (flat N(0,1.5^2), noise 0.5+0.1i, bias -1); c=0.35, T=768, Tm=1")
QWEN3_14B_SWEEP = Workload(
    "qwen3_14b_shape_B192_g16_V151936_d5120_bf16", B=192, gamma=16, V=151936, d=5120,
    dtype="bf16", temperature=0.7, cost_c=0.3, cap_T=1024, index=5, c_range=(0.1, 0.5),
    description="N(0,3^2) + U[2,12] spike per request, noise 0.05+U[0,0.4]+0.06i, "
                "c ~ U[0.1,0.5] per step, T=1024, Tm=0.7")

WORKLOADS = {w.name: w for w in (TINY, QWEN3_8B, LATENCY_B1, MIXED_B256, QWEN3_14B_SWEEP)}


def _normal(shape, std, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def _row_params(w: Workload, gen, device):
    """Per-request (background std, spike height, noise base, noise slope, bias)."""
    B = w.B
    ones = torch.ones(B, device=device)
    idx = w.index
    if idx == 1:
        return 2.0 * ones, 0.0 * ones, 0.2 * ones, 0.1 * ones, 1.0 * ones
    if idx == 2:
        return 3.0 * ones, 8.0 * ones, 0.3 * ones, 0.08 * ones, 0.0 * ones
    if idx == 3:
        return 2.0 * ones, 10.0 * ones, 0.1 * ones, 0.05 * ones, 0.0 * ones
    if idx == 4:
        code = torch.arange(B, device=device) < B // 2
        bg = torch.where(code, 2.0, 1.5).float()
        spike = torch.where(code, 10.0, 0.0).float()
        nb = torch.where(code, 0.1, 0.5).float()
        ns = torch.where(code, 0.04, 0.1).float()
        bias = torch.where(code, 2.0, -1.0).float()
        return bg, spike, nb, ns, bias
    if idx == 5:
        spike = 2.0 + 10.0 * torch.rand(B, generator=gen, device=device)
        nb = 0.05 + 0.4 * torch.rand(B, generator=gen, device=device)
        return 3.0 * ones, spike, nb, 0.06 * ones, 0.0 * ones
    raise ValueError(idx)


def _tau(w: Workload, device):
    i = torch.arange(w.gamma, device=device, dtype=torch.float32)
    if w.index == 1:
        return 1.0 + 0.05 * i
    if w.index == 2:
        return 1.0 + 0.03 * i
    return torch.ones(w.gamma, device=device)


def make_inputs(w: Workload, step: int = 0, device="cpu", temperature: Optional[float] = None,
                B: Optional[int] = None, V: Optional[int] = None, d: Optional[int] = None,
                gamma: Optional[int] = None, cap_T: Optional[int] = None,
                cost_c: Optional[float] = None, fixed_budget: int = -1,
                request_chunk: int = 16) -> dict:
    """Draw one step's inputs for workload ``w`` (optionally resized).

    Returns a dict of torch tensors on ``device`` plus Python scalars:
    hidden [B,gamma,d], head_w [d], head_bias [B], sts_tau [gamma],
    target_dense [B,gamma+1,V], draft_logits [B,gamma,V], draft_tokens
    [B,gamma] int32, last_tokens [B] int32, seq_lens [B] int32, cost_c,
    cap_T, temperature, seed, fixed_budget.
    """
    if B is not None or V is not None or d is not None or gamma is not None:
        w = dataclasses.replace(w, B=w.B if B is None else B, V=w.V if V is None else V,
                                d=w.d if d is None else d,
                                gamma=w.gamma if gamma is None else gamma)
    Tm = w.temperature if temperature is None else float(temperature)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + 100 * w.index + step)
    Bn, g, Vn, dn = w.B, w.gamma, w.V, w.d

    bg, spike, nb, ns, bias = _row_params(w, gen, device)
    hidden = _normal((Bn, g, dn), 1.0, gen, device).to(dt)
    head_w = _normal((dn,), 1.0 / math.sqrt(dn), gen, device)
    tau = _tau(w, device)
    if w.c_range is not None:
        lo, hi = w.c_range
        c = float(lo + (hi - lo) * torch.rand((), generator=gen, device=device).item())
    else:
        c = w.cost_c
    if cost_c is not None:
        c = float(cost_c)

    target = torch.empty((Bn, g + 1, Vn), dtype=dt, device=device)
    draft = torch.empty((Bn, g, Vn), dtype=dt, device=device)
    drafts = torch.empty((Bn, g), dtype=torch.int32, device=device)
    draw_T = w.draft_temperature if w.draft_temperature is not None else Tm
    pos = torch.arange(g, device=device, dtype=torch.float32)
    for b0 in range(0, Bn, request_chunk):
        b1 = min(Bn, b0 + request_chunk)
        nbk = b1 - b0
        t32 = _normal((nbk, g + 1, Vn), 1.0, gen, device) * bg[b0:b1, None, None]
        sp_idx = torch.randint(0, Vn, (nbk, g + 1), generator=gen, device=device)
        t32.scatter_add_(2, sp_idx[..., None],
                         spike[b0:b1, None, None].expand(nbk, g + 1, 1).contiguous())
        sigma = nb[b0:b1, None] + ns[b0:b1, None] * pos[None, :]
        q32 = t32[:, :g] + _normal((nbk, g, Vn), 1.0, gen, device) * sigma[..., None]
        target[b0:b1] = t32.to(dt)
        draft[b0:b1] = q32.to(dt)
        qd = draft[b0:b1].float()
        if draw_T > 0:
            u = torch.rand((nbk, g, Vn), generator=gen, device=device).clamp_(min=1e-20)
            gumbel = -torch.log(-torch.log(u))
            drafts[b0:b1] = torch.argmax(qd / draw_T + gumbel, dim=-1).to(torch.int32)
            del u, gumbel
        else:
            drafts[b0:b1] = torch.argmax(qd, dim=-1).to(torch.int32)
        del t32, q32, qd
    last = torch.randint(0, Vn, (Bn,), generator=gen, device=device, dtype=torch.int32)
    seq_lens = torch.randint(16, 4096, (Bn,), generator=gen, device=device, dtype=torch.int32)
    return {
        "workload": w.name, "B": Bn, "gamma": g, "V": Vn, "d": dn, "dtype": w.dtype,
        "hidden": hidden, "head_w": head_w.contiguous(), "head_bias": bias.contiguous(),
        "sts_tau": tau.contiguous(), "target_dense": target, "draft_logits": draft,
        "draft_tokens": drafts, "last_tokens": last, "seq_lens": seq_lens,
        "cost_c": float(c), "cap_T": int(w.cap_T if cap_T is None else cap_T),
        "temperature": float(Tm), "seed": int(step), "fixed_budget": int(fixed_budget),
    }


def to_numpy(inp: dict) -> dict:
    """Host numpy copies for the oracle: bf16 tensors become uint16 bit patterns."""
    out = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                out[k] = t.view(torch.int16).numpy().view("uint16")
            else:
                out[k] = t.numpy()
        else:
            out[k] = v
    return out


def ragged_target_rows(target_dense, row_req, row_k, n_rows: int):
    """Stand-in for the target forward over the packed rows: row r of the
    result is the target row (row_req[r], row_k[r]) of a dense
    [B, gamma+1, V] tensor.  A plain gather (torch), not part of the step."""
    B, g1, V = target_dense.shape
    idx = row_req[:n_rows].long() * g1 + row_k[:n_rows].long()
    return target_dense.reshape(B * g1, V).index_select(0, idx)
