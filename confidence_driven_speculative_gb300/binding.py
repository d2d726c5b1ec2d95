"""Thin ctypes binding of libdspark.so (include/dspark.h).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels behind the C ABI.  PyTorch provides device memory and the stream.
If the library has not been built this module raises; there is no fallback.

The three entry points keep their C names: :func:`dspark_score_budget`,
:func:`dspark_compact`, :func:`dspark_verify` (plus the workspace helpers);
:func:`dspark_score_compact` is the first two in one launch.
:class:`StepBuffers` allocates the caller-owned outputs and workspace of one
step shape and fills the ``dspark_step`` struct.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

DSPARK_OK, DSPARK_EINVAL, DSPARK_EDTYPE, DSPARK_EALIGN = 0, -1, -2, -3
DSPARK_ECUDA, DSPARK_EWORKSPACE, DSPARK_EDEVICE = -4, -5, -6
DSPARK_F32, DSPARK_BF16 = 0, 1
DSPARK_NO_CAP = -1
DSPARK_DYNAMIC = -1

_P = ctypes.c_void_p


class DsparkStep(ctypes.Structure):
    """Mirror of ``struct dspark_step`` (same field order and C types)."""
    _fields_ = [
        ("B", ctypes.c_int32), ("gamma", ctypes.c_int32), ("V", ctypes.c_int32),
        ("d", ctypes.c_int32), ("logit_dtype", ctypes.c_int32), ("hidden_dtype", ctypes.c_int32),
        ("draft_tokens", _P), ("draft_logits", _P), ("target_logits", _P), ("hidden", _P),
        ("head_w", _P), ("head_bias", _P), ("sts_tau", _P), ("last_tokens", _P),
        ("seq_lens_in", _P),
        ("cost_c", ctypes.c_float), ("cap_T", ctypes.c_int32), ("fixed_budget", ctypes.c_int32),
        ("temperature", ctypes.c_float), ("seed", ctypes.c_uint64),
        ("conf", _P), ("survival", _P), ("L0", _P), ("L", _P), ("draft_off", _P),
        ("row_off", _P), ("packed_ids", _P), ("packed_pos", _P), ("row_req", _P),
        ("row_k", _P), ("accept_len", _P), ("num_emitted", _P), ("out_tokens", _P),
        ("p_tok", _P), ("q_tok", _P), ("seq_lens_commit", _P),
        ("workspace", _P), ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libdspark.so (built by ``_build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        SP = ctypes.POINTER(DsparkStep)
        for name in ("dspark_score_budget", "dspark_score_compact", "dspark_compact",
                     "dspark_verify"):
            fn = getattr(lib, name)
            fn.argtypes = [SP, _P]
            fn.restype = ctypes.c_int
        lib.dspark_fit_sts_tau.argtypes = [ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P,
                                           ctypes.c_float, ctypes.c_float, _P, _P, _P, _P]
        lib.dspark_fit_sts_tau.restype = ctypes.c_int
        lib.dspark_score_entropy.argtypes = [SP, ctypes.c_float, _P]
        lib.dspark_score_entropy.restype = ctypes.c_int
        lib.dspark_verify_cap_accept.argtypes = [SP, _P, _P, _P, _P]
        lib.dspark_verify_cap_accept.restype = ctypes.c_int
        lib.dspark_verify_noalloc.argtypes = [SP, ctypes.c_int32, _P, _P]
        lib.dspark_verify_noalloc.restype = ctypes.c_int
        lib.dspark_workspace_size.argtypes = [ctypes.c_int32] * 4
        lib.dspark_workspace_size.restype = ctypes.c_size_t
        lib.dspark_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
        lib.dspark_workspace_init.restype = ctypes.c_int
        lib.dspark_read_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
        lib.dspark_read_device_status.restype = ctypes.c_int
        lib.dspark_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.dspark_set_wait_timeout_ns.restype = ctypes.c_int
        lib.dspark_wait_timeout_ns.argtypes = []
        lib.dspark_wait_timeout_ns.restype = ctypes.c_uint64
        lib.dspark_last_error.argtypes = []
        lib.dspark_last_error.restype = ctypes.c_char_p
        lib.dspark_version.argtypes = []
        lib.dspark_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


class DsparkError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what} returned {status}: {last_error()}")
        self.status = status


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream)


def _call(name: str, step: DsparkStep, stream, check: bool) -> int:
    rc = getattr(load(), name)(ctypes.byref(step), _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, name)
    return rc


def dspark_score_budget(step: DsparkStep, stream=None, check: bool = True) -> int:
    return _call("dspark_score_budget", step, stream, check)


def dspark_score_entropy(step: DsparkStep, theta: float, stream=None, check: bool = True) -> int:
    """Steps a1-a3 with conf = exp(-entropy of softmax(draft logits / theta))."""
    rc = load().dspark_score_entropy(ctypes.byref(step), float(theta), _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_score_entropy")
    return rc


def dspark_compact(step: DsparkStep, stream=None, check: bool = True) -> int:
    return _call("dspark_compact", step, stream, check)


def dspark_score_compact(step: DsparkStep, stream=None, check: bool = True) -> int:
    """dspark_score_budget then dspark_compact, in one kernel launch."""
    return _call("dspark_score_compact", step, stream, check)


def dspark_verify(step: DsparkStep, stream=None, check: bool = True) -> int:
    return _call("dspark_verify", step, stream, check)


def dspark_verify_cap_accept(step: DsparkStep, commit_len, accept_full=None, audit_totals=None,
                             stream=None, check: bool = True) -> int:
    """The cap-accept audit arm: verify the step's full block, commit the
    window ``commit_len`` (device int32 [B]).  ``accept_full`` (device int32
    [B]) and ``audit_totals`` (device int32 [2]) are optional outputs."""
    B = int(step.B)
    _device_array(commit_len, "commit_len", "int32", B)
    _device_array(accept_full, "accept_full", "int32", B, optional=True)
    _device_array(audit_totals, "audit_totals", "int32", 2, optional=True)
    rc = load().dspark_verify_cap_accept(ctypes.byref(step), _ptr(commit_len), _ptr(accept_full),
                                         _ptr(audit_totals), _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_verify_cap_accept")
    return rc


def dspark_fit_sts_tau(conf, tau_used, L, accept_len, tau_out, tau_min: float = 0.05,
                       tau_max: float = 20.0, nll_out=None, n_obs=None, stream=None,
                       check: bool = True) -> int:
    """STS temperatures fitted to logged steps (device tensors: conf [N, gamma]
    float32, tau_used [gamma] float32, L / accept_len [N] int32; writes
    tau_out [gamma], and nll_out / n_obs when given)."""
    if conf is None or conf.dim() != 2:
        raise ValueError("conf must be a [N, gamma] tensor")
    N, gamma = int(conf.shape[0]), int(conf.shape[1])
    if N > 0:
        _device_array(conf, "conf", "float32")
        _device_array(L, "L", "int32", N)
        _device_array(accept_len, "accept_len", "int32", N)
    _device_array(tau_used, "tau_used", "float32", gamma)
    _device_array(tau_out, "tau_out", "float32", gamma)
    _device_array(nll_out, "nll_out", "float32", gamma, optional=True)
    _device_array(n_obs, "n_obs", "int32", gamma, optional=True)
    rc = load().dspark_fit_sts_tau(N, gamma, _ptr(conf), _ptr(tau_used), _ptr(L),
                                   _ptr(accept_len), float(tau_min), float(tau_max),
                                   _ptr(tau_out), _ptr(nll_out), _ptr(n_obs), _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_fit_sts_tau")
    return rc


DSPARK_NOALLOC_SCRATCH_BYTES = 8 << 20


def dspark_verify_noalloc(step: DsparkStep, reset: bool = False, status_out=None, stream=None,
                          check: bool = True) -> int:
    """dspark_verify on the library's fixed scratch (no workspace, no device
    allocation); ``step.workspace`` is ignored.  ``status_out`` is a device
    int32 tensor or None."""
    rc = load().dspark_verify_noalloc(ctypes.byref(step), int(bool(reset)), _ptr(status_out),
                                      _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_verify_noalloc")
    return rc


def dspark_workspace_size(B: int, gamma: int, V: int, d: int) -> int:
    return int(load().dspark_workspace_size(B, gamma, V, d))


def dspark_workspace_init(ptr: int, nbytes: int, stream=None, check: bool = True) -> int:
    rc = load().dspark_workspace_init(ptr, nbytes, _stream(stream))
    if check and rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_workspace_init")
    return rc


def dspark_read_device_status(ptr: int, stream=None) -> int:
    out = ctypes.c_int32(-1)
    rc = load().dspark_read_device_status(ptr, ctypes.byref(out), _stream(stream))
    if rc != DSPARK_OK:
        raise DsparkError(rc, "dspark_read_device_status")
    return int(out.value)


def dspark_set_wait_timeout_ns(ns: int) -> int:
    """Bound of every device wait in later launches (0: the 2 s default)."""
    return int(load().dspark_set_wait_timeout_ns(int(ns)))


def dspark_wait_timeout_ns() -> int:
    return int(load().dspark_wait_timeout_ns())


def last_error() -> str:
    return load().dspark_last_error().decode()


def version() -> str:
    return load().dspark_version().decode()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DSPARK_F32
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _device_array(t, name: str, dtype: str, numel: Optional[int] = None, optional=False):
    """Check that ``t`` is a contiguous CUDA tensor of ``dtype`` ("int32" or
    "float32") with ``numel`` elements (when given); raise ValueError
    otherwise, before anything reaches the library."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    import torch
    want = {"int32": torch.int32, "float32": torch.float32}[dtype]
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.dtype != want:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be CUDA device memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


class StepBuffers:
    """Caller-owned device outputs and workspace for one step shape, plus the
    ``dspark_step`` struct pointing at them.  Inputs are attached with
    :meth:`bind`; the ragged target rows with :meth:`bind_target`."""

    def __init__(self, B: int, gamma: int, V: int, d: int, device="cuda", stream=None):
        import torch
        self.B, self.gamma, self.V, self.d = B, gamma, V, d
        i32, f32 = torch.int32, torch.float32
        cap = max(B * (gamma + 1), 1)
        kw = dict(device=device)
        self.conf = torch.zeros((B, gamma), dtype=f32, **kw)
        self.survival = torch.zeros((B, gamma), dtype=f32, **kw)
        self.L0 = torch.zeros(B, dtype=i32, **kw)
        self.L = torch.zeros(B, dtype=i32, **kw)
        self.draft_off = torch.zeros(B + 1, dtype=i32, **kw)
        self.row_off = torch.zeros(B + 1, dtype=i32, **kw)
        self.packed_ids = torch.zeros(cap, dtype=i32, **kw)
        self.packed_pos = torch.zeros(cap, dtype=i32, **kw)
        self.row_req = torch.zeros(cap, dtype=i32, **kw)
        self.row_k = torch.zeros(cap, dtype=i32, **kw)
        self.accept_len = torch.zeros(B, dtype=i32, **kw)
        self.num_emitted = torch.zeros(B, dtype=i32, **kw)
        self.out_tokens = torch.zeros((B, gamma + 1), dtype=i32, **kw)
        self.p_tok = torch.zeros(max(B * gamma, 1), dtype=f32, **kw)
        self.q_tok = torch.zeros(max(B * gamma, 1), dtype=f32, **kw)
        self.ws_bytes = dspark_workspace_size(B, gamma, V, d)
        if self.ws_bytes == 0:
            raise ValueError("shape outside the library's limits")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, **kw)
        assert self.workspace.data_ptr() % 256 == 0
        dspark_workspace_init(self.workspace.data_ptr(), self.ws_bytes, stream)
        self.step = DsparkStep()
        s = self.step
        s.B, s.gamma, s.V, s.d = B, gamma, V, d
        for name in ("conf", "survival", "L0", "L", "draft_off", "row_off", "packed_ids",
                     "packed_pos", "row_req", "row_k", "accept_len", "num_emitted",
                     "out_tokens", "p_tok", "q_tok"):
            setattr(s, name, getattr(self, name).data_ptr())
        s.workspace = self.workspace.data_ptr()
        s.workspace_bytes = self.ws_bytes
        s.fixed_budget = DSPARK_DYNAMIC
        s.cap_T = DSPARK_NO_CAP
        self._keep = {}

    def bind(self, inp: dict, seq_lens_commit=None) -> "StepBuffers":
        """Point the struct at a dict of device inputs (as made by
        :func:`workloads.make_inputs`)."""
        s = self.step
        keep = self._keep
        keep.clear()
        for k in ("draft_tokens", "draft_logits", "hidden", "head_w", "head_bias", "sts_tau",
                  "last_tokens", "seq_lens"):
            keep[k] = inp.get(k)
        s.logit_dtype = _dtype_code(inp["draft_logits"])
        s.hidden_dtype = _dtype_code(inp["hidden"])
        s.draft_tokens = _ptr(inp["draft_tokens"])
        s.draft_logits = _ptr(inp["draft_logits"])
        s.hidden = _ptr(inp["hidden"])
        s.head_w = _ptr(inp["head_w"])
        s.head_bias = _ptr(inp["head_bias"])
        s.sts_tau = _ptr(inp["sts_tau"])
        s.last_tokens = _ptr(inp.get("last_tokens"))
        s.seq_lens_in = _ptr(inp.get("seq_lens"))
        s.cost_c = float(inp["cost_c"])
        s.cap_T = int(inp["cap_T"])
        s.fixed_budget = int(inp.get("fixed_budget", -1))
        s.temperature = float(inp["temperature"])
        s.seed = int(inp["seed"])
        keep["seq_lens_commit"] = seq_lens_commit
        s.seq_lens_commit = _ptr(seq_lens_commit)
        return self

    def bind_target(self, target_ragged) -> "StepBuffers":
        self._keep["target"] = target_ragged
        self.step.target_logits = _ptr(target_ragged)
        return self

    def device_status(self, stream=None) -> int:
        return dspark_read_device_status(self.workspace.data_ptr(), stream)
