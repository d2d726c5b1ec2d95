"""Plain fp64 CPU oracle for the confidence-driven variable-length verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
calls it, and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain loops, double precision); this
module compiles it with gcc and marshals numpy arrays through ctypes.  Array
conventions:

* logits and hidden states are numpy ``float32`` (fp32) or ``uint16`` holding
  bfloat16 bit patterns (bf16);
* integer arrays are ``int32``; every float output is ``float64``.

Function-to-source map (page titles and sections):

* :func:`philox4x64_10`, :func:`uniforms` -- Salmon et al., SC'11, Philox4x64-10.
* :func:`score` -- "DFlash to DSpark in SGLang", section "DSpark: a sequential
  head and a verify budget" (confidence head, STS, survival, budget rule).
* :func:`score_entropy` -- "SGLang Integrates DSpark ...", section "DSpark's
  Core Idea: Only Verify the Parts You're Confident About" (confidence from
  the entropy of the drafter's distribution); survival and budget as above.
* :func:`fit_sts_tau` -- "DFlash to DSpark in SGLang", "DSpark: a sequential
  head and a verify budget" (STS calibrates the survival to acceptance).
* :func:`cap` -- same page, section "Zero-overhead scheduling and kernels"
  (verify-length top-k schedule under a batch-wide cap).
* :func:`fixed_budget` -- same page, "The confidence scheduler and verify modes".
* :func:`compact` -- same page, "Ragged verify under full CUDA graphs".
* :func:`verify`, :func:`verify_request` -- same page, "Background"; and
  "SGLang Integrates DSpark ...", section "The Old Problem with Speculative
  Decoding: It Breaks Down at Scale" (speculative sampling).
* :func:`verify_cap_accept` -- "DFlash to DSpark in SGLang", "The confidence
  scheduler and verify modes" (the cap-accept audit arm) and "Scheduling
  results" (utilization against the ceiling).

Parity pins for every function are in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_OMP_PATH = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_omp = None

F32, BF16 = 0, 1


def _compile(path: str, extra, force: bool) -> str:
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", *extra,
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False, omp: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2); with
    ``omp`` also ``liboracle_omp.so``, the same source with its OpenMP batch
    verify enabled (for the benchmark's multi-core CPU baseline)."""
    path = _compile(_LIB_PATH, [], force)
    if omp:
        _compile(_OMP_PATH, ["-fopenmp", "-DORC_OMP"], force)
    return path


def _load_omp():
    """The OpenMP build: only its batch verify is used."""
    global _omp
    with _lock:
        if _omp is None:
            build(omp=True)
            lib = ctypes.CDLL(_OMP_PATH)
            P = ctypes.c_void_p
            i32, f64, u64 = ctypes.c_int, ctypes.c_double, ctypes.c_uint64
            lib.orc_verify_omp.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, f64, u64, f64,
                                           f64, f64, P, P, P, P, P, P, P]
            lib.orc_verify_omp.restype = ctypes.c_int
            lib.orc_omp_threads.argtypes = [i32]
            lib.orc_omp_threads.restype = ctypes.c_int
            _omp = lib
    return _omp


def omp_threads(n: int = 0) -> int:
    """Threads the OpenMP batch verify uses (n > 0 sets them)."""
    return int(_load_omp().orc_omp_threads(int(n)))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, f64, u64, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_int64
            lib.orc_philox4x64_10.argtypes = [P, P, P]
            lib.orc_philox4x64_10.restype = None
            lib.orc_uniforms.argtypes = [u64, i64, i64, P, P, P]
            lib.orc_uniforms.restype = None
            lib.orc_score.argtypes = [i32, i32, i32, i32, P, P, P, P, f64, f64, P, P, P, P]
            lib.orc_score_entropy.argtypes = [i32, i32, i32, i32, P, f64, f64, f64, P, P, P, P]
            lib.orc_fit_sts_tau.argtypes = [i32, i32, P, P, P, P, f64, f64, P, P, P]
            lib.orc_fixed_budget.argtypes = [i32, i32, i32, P]
            lib.orc_cap.argtypes = [i32, i32, P, P, i32, f64, P, P]
            lib.orc_compact.argtypes = [i32, i32, P, P, P, P, P, P, P, P, P, P]
            lib.orc_verify_request.argtypes = [i32, i32, i32, P, P, P, f64, P, P, P, f64, f64,
                                               f64, P, P, P, P, P]
            lib.orc_check_request.argtypes = [i32, i32, i32, P, P, P, f64, P, P, P, f64, f64,
                                              f64, i32, i32, P, P]
            lib.orc_verify.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, f64, u64, f64, f64,
                                       f64, P, P, P, P, P, P, P]
            for name in ("orc_score", "orc_score_entropy", "orc_fit_sts_tau",
                         "orc_fixed_budget", "orc_cap",
                         "orc_compact", "orc_verify_request", "orc_verify"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logit_dtype(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits/hidden must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def philox4x64_10(ctr, key) -> np.ndarray:
    """One Philox4x64-10 block: four 64-bit words for counter ``ctr`` (4 words), key ``key`` (2)."""
    lib = _load()
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib.orc_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, b: int, k: int) -> tuple[float, float, float]:
    """(u, u', u'') of draft position ``k`` of request ``b``: words 0, 1, 2 of
    Philox counter (b,k,0,0), key (seed,0)."""
    lib = _load()
    u = ctypes.c_double()
    u2 = ctypes.c_double()
    u3 = ctypes.c_double()
    lib.orc_uniforms(ctypes.c_uint64(seed), b, k, ctypes.byref(u), ctypes.byref(u2),
                     ctypes.byref(u3))
    return u.value, u2.value, u3.value


def score(hidden, w, bias, tau, c: float, eps: float = 1e-5):
    """Confidence head + STS + survival + pre-cap budget.

    ``hidden`` [B, gamma, d]; ``w`` [d]; ``bias`` [B]; ``tau`` [gamma].
    Returns ``(conf [B,gamma], surv [B,gamma] (S_1..S_gamma), L0 [B], tie [B])``.
    """
    lib = _load()
    hidden = np.ascontiguousarray(hidden)
    B, gamma, d = hidden.shape
    w = _c(w, np.float32)
    bias = _c(bias, np.float32)
    tau = _c(tau, np.float32)
    conf = np.zeros((B, gamma), np.float64)
    surv = np.zeros((B, gamma), np.float64)
    L0 = np.zeros(B, np.int32)
    tie = np.zeros(B, np.int32)
    rc = lib.orc_score(B, gamma, d, _logit_dtype(hidden), _ptr(hidden), _ptr(w), _ptr(bias),
                       _ptr(tau), float(np.float32(c)), eps, _ptr(conf), _ptr(surv), _ptr(L0),
                       _ptr(tie))
    _check(rc, "score")
    return conf, surv, L0, tie


def score_entropy(draft_logits, theta: float, c: float, eps: float = 1e-5):
    """Entropy confidence + survival + pre-cap budget.

    ``draft_logits`` [B, gamma, V]; ``theta`` the temperature of the
    drafter's distribution q = softmax(z_q / theta).  conf = exp(-H(q)).
    Returns ``(conf, surv, L0, tie)`` as :func:`score`.
    """
    lib = _load()
    z = np.ascontiguousarray(draft_logits)
    B, gamma, V = z.shape
    conf = np.zeros((B, gamma), np.float64)
    surv = np.zeros((B, gamma), np.float64)
    L0 = np.zeros(B, np.int32)
    tie = np.zeros(B, np.int32)
    rc = lib.orc_score_entropy(B, gamma, V, _logit_dtype(z), _ptr(z), float(np.float32(theta)),
                               float(np.float32(c)), eps, _ptr(conf), _ptr(surv), _ptr(L0),
                               _ptr(tie))
    _check(rc, "score_entropy")
    return conf, surv, L0, tie


def fit_sts_tau(conf, tau_used, L, accept_len, tau_min: float = 0.05,
                tau_max: float = 20.0):
    """Per-position STS temperatures by maximum likelihood on logged steps.

    ``conf`` [N, gamma] confidences a step produced with temperatures
    ``tau_used`` [gamma]; ``L`` [N] verify lengths; ``accept_len`` [N].
    Returns ``(tau [gamma], nll [gamma], n_obs [gamma])``.
    """
    lib = _load()
    conf = _c(conf, np.float32)
    N, gamma = conf.shape
    tau_used = _c(tau_used, np.float32)
    L = _c(L, np.int32)
    a = _c(accept_len, np.int32)
    tau = np.zeros(gamma, np.float64)
    nll = np.zeros(gamma, np.float64)
    nobs = np.zeros(gamma, np.int32)
    rc = lib.orc_fit_sts_tau(N, gamma, _ptr(conf), _ptr(tau_used), _ptr(L), _ptr(a),
                             float(np.float32(tau_min)), float(np.float32(tau_max)), _ptr(tau),
                             _ptr(nll), _ptr(nobs))
    _check(rc, "fit_sts_tau")
    return tau, nll, nobs


def fixed_budget(B: int, gamma: int, F: int) -> np.ndarray:
    lib = _load()
    L = np.zeros(B, np.int32)
    _check(lib.orc_fixed_budget(B, gamma, F, _ptr(L)), "fixed_budget")
    return L


def cap(surv, L0, T: int, eps: float = 2e-5):
    """Top-T cap over marginal gains. ``surv`` [B, gamma] (S_1..S_gamma). Returns ``(L, tie)``."""
    lib = _load()
    surv = _c(surv, np.float64)
    L0 = _c(L0, np.int32)
    B, gamma = surv.shape
    L = np.zeros(B, np.int32)
    tie = ctypes.c_int32()
    rc = lib.orc_cap(B, gamma, _ptr(surv), _ptr(L0), int(T), eps, _ptr(L), ctypes.byref(tie))
    _check(rc, "cap")
    return L, int(tie.value)


def compact(L, draft_tokens, last_tokens=None, seq_lens=None) -> dict:
    """Exclusive scans and ragged packing. ``draft_tokens`` [B, gamma]."""
    lib = _load()
    L = _c(L, np.int32)
    draft_tokens = _c(draft_tokens, np.int32)
    B, gamma = draft_tokens.shape
    last_tokens = None if last_tokens is None else _c(last_tokens, np.int32)
    seq_lens = None if seq_lens is None else _c(seq_lens, np.int32)
    cap_rows = B * (gamma + 1)
    out = {
        "draft_off": np.zeros(B + 1, np.int32),
        "row_off": np.zeros(B + 1, np.int32),
        "packed_ids": np.zeros(cap_rows, np.int32),
        "packed_pos": np.zeros(cap_rows, np.int32),
        "row_req": np.zeros(cap_rows, np.int32),
        "row_k": np.zeros(cap_rows, np.int32),
    }
    rc = lib.orc_compact(B, gamma, _ptr(L), _ptr(draft_tokens), _ptr(last_tokens),
                         _ptr(seq_lens), _ptr(out["draft_off"]), _ptr(out["row_off"]),
                         _ptr(out["packed_ids"]), _ptr(out["packed_pos"]), _ptr(out["row_req"]),
                         _ptr(out["row_k"]))
    _check(rc, "compact")
    return out


EPS_U, EPS_BLK, EPS_TOK = 1e-5, 1e-6, 2e-6


def verify_request(L: int, drafts, tgt, dft, Tm: float, u, u2, u3, eps: float = EPS_U,
                   eps_blk: float = EPS_BLK, eps_tok: float = EPS_TOK):
    """Verify one request with explicit uniforms.

    ``tgt`` [L+1, V] target rows (root first), ``dft`` [L, V] draft rows (may be
    ``None`` when ``Tm == 0``), ``u``/``u2``/``u3`` [L+1] (accept, block,
    in-block).  Returns ``(a, token, p[L], q[L], tie)``.
    """
    lib = _load()
    tgt = np.ascontiguousarray(tgt)
    V = tgt.shape[-1]
    if dft is None:
        dft = np.zeros((max(L, 1), V), tgt.dtype)
    dft = np.ascontiguousarray(dft, dtype=tgt.dtype)
    drafts = _c(drafts, np.int32) if L > 0 else np.zeros(1, np.int32)
    u = _c(u, np.float64)
    u2 = _c(u2, np.float64)
    u3 = _c(u3, np.float64)
    a = ctypes.c_int32()
    tok = ctypes.c_int32()
    tie = ctypes.c_int32()
    p = np.zeros(max(L, 1), np.float64)
    q = np.zeros(max(L, 1), np.float64)
    rc = lib.orc_verify_request(L, V, _logit_dtype(tgt), _ptr(drafts), _ptr(tgt), _ptr(dft),
                                float(np.float32(Tm)), _ptr(u), _ptr(u2), _ptr(u3), eps,
                                eps_blk, eps_tok, ctypes.byref(a),
                                ctypes.byref(tok), _ptr(p), _ptr(q), ctypes.byref(tie))
    _check(rc, "verify_request")
    return int(a.value), int(tok.value), p[:L], q[:L], int(tie.value)


def check_request(L: int, drafts, tgt, dft, Tm: float, u, u2, u3, a_g: int, tok_g: int,
                  eps: float = EPS_U, eps_blk: float = EPS_BLK, eps_tok: float = EPS_TOK):
    """Is ``(a_g, tok_g)`` an outcome this request admits once every decision
    within its tolerance window may go either way?  Arguments as
    :func:`verify_request`.  Returns ``(verdict, kinds)``: verdict 0 when
    admitted (else 1 a out of range, 2 an earlier test rejects outside its
    window, 3 the test at a accepts outside its window, 4 the token is not an
    outcome of the draw at row a, 5 greedy mismatch; ``tok_g`` < 0 checks the
    accept length alone); ``kinds`` counts the
    open decisions on the outcome's path: accept tests, residual masses
    below eps, draws with a near tie."""
    lib = _load()
    tgt = np.ascontiguousarray(tgt)
    V = tgt.shape[-1]
    if dft is None:
        dft = np.zeros((max(L, 1), V), tgt.dtype)
    dft = np.ascontiguousarray(dft, dtype=tgt.dtype)
    drafts = _c(drafts, np.int32)
    if drafts.size == 0:
        drafts = np.zeros(1, np.int32)
    u, u2, u3 = (_c(x, np.float64) for x in (u, u2, u3))
    kinds = np.zeros(3, np.int32)
    verdict = ctypes.c_int32(-1)
    rc = lib.orc_check_request(L, V, _logit_dtype(tgt), _ptr(drafts), _ptr(tgt), _ptr(dft),
                               float(np.float32(Tm)), _ptr(u), _ptr(u2), _ptr(u3), eps, eps_blk,
                               eps_tok, int(a_g), int(tok_g), _ptr(kinds), ctypes.byref(verdict))
    _check(rc, "check_request")
    return int(verdict.value), kinds


def verify(draft_tokens, draft_logits, target_ragged, L, row_off, draft_off, Tm: float,
           seed: int, eps: float = EPS_U, seq_lens=None, eps_blk: float = EPS_BLK,
           eps_tok: float = EPS_TOK, threads: int = 1) -> dict:
    """Verify the batch.

    ``draft_logits`` [B, gamma, V]; ``target_ragged`` [N_rows, V] with request
    b's rows at ``row_off[b] .. row_off[b] + L[b]``.  ``threads`` > 1 runs the
    requests on that many host threads (the OpenMP build; same results).
    """
    lib = _load()
    draft_tokens = _c(draft_tokens, np.int32)
    B, gamma = draft_tokens.shape
    target_ragged = np.ascontiguousarray(target_ragged)
    dt = _logit_dtype(target_ragged)
    V = target_ragged.shape[-1]
    draft_logits = np.ascontiguousarray(draft_logits, dtype=target_ragged.dtype)
    L = _c(L, np.int32)
    row_off = _c(row_off, np.int32)
    draft_off = _c(draft_off, np.int32)
    nL = int(draft_off[B]) if B > 0 else 0
    out = {
        "accept_len": np.zeros(B, np.int32),
        "num_emitted": np.zeros(B, np.int32),
        "out_tokens": np.zeros((B, gamma + 1), np.int32),
        "p_tok": np.zeros(max(nL, 1), np.float64),
        "q_tok": np.zeros(max(nL, 1), np.float64),
        "tie": np.zeros(B, np.int32),
    }
    sl = None if seq_lens is None else _c(seq_lens, np.int32).copy()
    fn = lib.orc_verify
    if threads > 1:
        omp_threads(threads)
        fn = _load_omp().orc_verify_omp
    rc = fn(B, gamma, V, dt, _ptr(draft_tokens), _ptr(draft_logits),
                        _ptr(target_ragged), _ptr(L), _ptr(row_off), _ptr(draft_off),
                        float(np.float32(Tm)), ctypes.c_uint64(seed), eps, eps_blk, eps_tok,
                        _ptr(out["accept_len"]), _ptr(out["num_emitted"]), _ptr(out["out_tokens"]),
                        _ptr(out["p_tok"]), _ptr(out["q_tok"]), _ptr(sl), _ptr(out["tie"]))
    _check(rc, "verify")
    out["p_tok"] = out["p_tok"][:nL]
    out["q_tok"] = out["q_tok"][:nL]
    if sl is not None:
        out["seq_lens"] = sl
    return out


def ragged_target(target_dense, L, row_off) -> np.ndarray:
    """Stand-in for the target forward: the ragged rows [root, d_1..d_L] of each
    request, copied out of a dense [B, gamma+1, V] array of target logits."""
    target_dense = np.asarray(target_dense)
    B = target_dense.shape[0]
    V = target_dense.shape[-1]
    n = int(row_off[B]) if B > 0 else 0
    out = np.empty((max(n, 1), V), target_dense.dtype)
    for b in range(B):
        out[row_off[b]:row_off[b] + L[b] + 1] = target_dense[b, :L[b] + 1]
    return out[:n] if n > 0 else out[:0]


def step(inp: dict, eps_s: float = 1e-5, eps_cap: float = 2e-5, eps_u: float = EPS_U,
         L_override=None, threads: int = 1) -> dict:
    """The whole step a1..a6 on one input dict (keys as produced by the
    workload generators): score, cap (or fixed budget), compact, the
    target-forward stand-in, verify.  ``L_override`` replaces the computed
    verify lengths (used when a flagged near tie was decided the other way by
    a reduced-precision implementation)."""
    B, gamma = inp["draft_tokens"].shape
    res = {}
    fixed = inp.get("fixed_budget", -1)
    if fixed is not None and fixed >= 0:
        L = fixed_budget(B, gamma, fixed)
        res["score_tie"] = np.zeros(B, np.int32)
        res["cap_tie"] = 0
    else:
        conf, surv, L0, tie = score(inp["hidden"], inp["head_w"], inp["head_bias"],
                                    inp["sts_tau"], inp["cost_c"], eps_s)
        L, cap_tie = cap(surv, L0, inp["cap_T"], eps_cap)
        res.update(conf=conf, surv=surv, L0=L0, score_tie=tie, cap_tie=cap_tie)
    if L_override is not None:
        L = np.asarray(L_override, np.int32)
    res["L"] = L
    res.update(compact(L, inp["draft_tokens"], inp.get("last_tokens"), inp.get("seq_lens")))
    tgt = ragged_target(inp["target_dense"], L, res["row_off"])
    v = verify(inp["draft_tokens"], inp["draft_logits"], tgt, L, res["row_off"],
               res["draft_off"], inp["temperature"], inp["seed"], eps_u, inp.get("seq_lens"),
               threads=threads)
    res.update(v)
    return res


def verify_cap_accept(draft_tokens, draft_logits, target_dense, L, W, Tm: float, seed: int,
                      eps: float = EPS_U, seq_lens=None) -> dict:
    """The cap-accept audit arm: verify the full block, commit only the window.

    "DFlash to DSpark in SGLang", "The confidence scheduler and verify modes":
    cap-accept pays the verify cost of the full block ``L`` (static: every
    L_b = gamma) but commits what compact would commit with window ``W``, and
    records what the trim gave up.  Written as its definition: two plain
    verifies on the same target and draft logits and the same Philox stream.

    * the full verify over ``L`` gives ``accept_full`` (the ceiling a_full)
      and the per-draft ``p_tok`` / ``q_tok`` of the full layout;
    * the window verify over ``min(max(W, 0), L)`` gives every committed
      output (``accept_len``, ``num_emitted``, ``out_tokens``, ``seq_lens``).

    ``audit_totals`` = (sum of a_full, sum of committed accept_len).  Their
    ratio is the utilization against the ceiling of "Scheduling results",
    read here as accepted drafts kept / accepted drafts a full verify finds.
    ``tie`` flags a near tie in either verify.  ``target_dense`` is
    [B, gamma+1, V]; both layouts are cut from it with :func:`ragged_target`.
    """
    draft_tokens = _c(draft_tokens, np.int32)
    B, gamma = draft_tokens.shape
    L = np.clip(_c(L, np.int32), 0, gamma).astype(np.int32)
    Wc = np.minimum(np.maximum(_c(W, np.int32), 0), L).astype(np.int32)
    full_lay = compact(L, draft_tokens)
    full = verify(draft_tokens, draft_logits, ragged_target(target_dense, L, full_lay["row_off"]),
                  L, full_lay["row_off"], full_lay["draft_off"], Tm, seed, eps)
    win_lay = compact(Wc, draft_tokens)
    win = verify(draft_tokens, draft_logits, ragged_target(target_dense, Wc, win_lay["row_off"]),
                 Wc, win_lay["row_off"], win_lay["draft_off"], Tm, seed, eps, seq_lens)
    out = {k: win[k] for k in ("accept_len", "num_emitted", "out_tokens")}
    if "seq_lens" in win:
        out["seq_lens"] = win["seq_lens"]
    out["accept_full"] = full["accept_len"]
    out["p_tok"] = full["p_tok"]
    out["q_tok"] = full["q_tok"]
    out["tie"] = (full["tie"] | win["tie"]).astype(np.int32)
    out["W"] = Wc
    out["audit_totals"] = np.array([int(full["accept_len"].sum()), int(win["accept_len"].sum())],
                                   np.int64)
    return out
