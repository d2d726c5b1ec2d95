"""CPU checks of the C ABI: the library builds for sm_103a, exports every
function include/dspark.h declares, the ctypes struct matches the C layout, and
host-side validation returns the documented codes before touching the GPU."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from confidence_driven_speculative_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_step_calls():
    names = declared_functions()
    for n in ("dspark_score_budget", "dspark_compact", "dspark_verify",
              "dspark_workspace_size", "dspark_workspace_init", "dspark_last_error"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing
    out = subprocess.run(["nm", "-D", "--defined-only", binding.lib_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dspark_\w+)", out))
    assert set(declared_functions()) <= exported


def test_struct_layout_matches_c(lib):
    fields = [f for f, _ in binding.DsparkStep._fields_]
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "dspark.h"', "int main(void){",
           'printf("%zu\\n", sizeof(dspark_step));']
    src += [f'printf("%zu\\n", offsetof(dspark_step, {f}));' for f in fields]
    src += ["return 0;}"]
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "layout.c")
        exe = os.path.join(td, "layout")
        open(c, "w").write("\n".join(src))
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(binding.DsparkStep)
    for f, off in zip(fields, vals[1:]):
        assert getattr(binding.DsparkStep, f).offset == off, f


def test_workspace_size(lib):
    assert binding.dspark_workspace_size(256, 16, 129280, 7168) > 0
    assert binding.dspark_workspace_size(0, 16, 129280, 7168) > 0
    assert binding.dspark_workspace_size(-1, 16, 10, 10) == 0
    assert binding.dspark_workspace_size(4, 0, 10, 10) == 0
    assert binding.dspark_workspace_size(4, 65, 10, 10) == 0
    assert binding.dspark_workspace_size(4, 8, 0, 10) == 0
    a = binding.dspark_workspace_size(64, 16, 129280, 7168)
    b = binding.dspark_workspace_size(128, 16, 129280, 7168)
    assert b > a and a % 256 == 0 and b % 256 == 0


FAKE = 1 << 20  # a 256-aligned non-null address; validation never dereferences it


def valid_step(B=4, gamma=8, V=1024, d=256):
    s = binding.DsparkStep()
    s.B, s.gamma, s.V, s.d = B, gamma, V, d
    s.logit_dtype = s.hidden_dtype = binding.DSPARK_BF16
    for name, _ in binding.DsparkStep._fields_:
        if isinstance(getattr(s, name), (int, type(None))) and name not in (
                "B", "gamma", "V", "d", "logit_dtype", "hidden_dtype", "cap_T", "fixed_budget",
                "seed", "workspace_bytes"):
            setattr(s, name, FAKE)
    s.cap_T = binding.DSPARK_NO_CAP
    s.fixed_budget = binding.DSPARK_DYNAMIC
    s.cost_c = 0.3
    s.temperature = 1.0
    s.workspace_bytes = binding.dspark_workspace_size(B, gamma, V, d)
    return s


CALLS = ["dspark_score_budget", "dspark_score_compact", "dspark_compact", "dspark_verify"]


@pytest.mark.parametrize("call", CALLS)
def test_null_step_and_bad_shapes(lib, call):
    fn = getattr(lib, call)
    assert fn(None, None) == binding.DSPARK_EINVAL
    assert "NULL" in binding.last_error()
    for field, val in [("B", -1), ("B", 65537), ("gamma", 0), ("gamma", 65), ("V", 0), ("d", 0)]:
        s = valid_step()
        setattr(s, field, val)
        assert fn(ctypes.byref(s), None) == binding.DSPARK_EINVAL, (field, val)
    s = valid_step()
    s.logit_dtype = 7
    assert fn(ctypes.byref(s), None) == binding.DSPARK_EDTYPE
    s = valid_step()
    s.hidden_dtype = -3
    assert fn(ctypes.byref(s), None) == binding.DSPARK_EDTYPE


@pytest.mark.parametrize("call", CALLS)
def test_empty_batch_is_a_no_op(lib, call):
    s = valid_step(B=0)
    assert getattr(lib, call)(ctypes.byref(s), None) == binding.DSPARK_OK


@pytest.mark.parametrize("call", ["dspark_score_budget", "dspark_score_compact"])
def test_score_budget_validation(lib, call):
    f = getattr(lib, call)
    s = valid_step(); s.L = None
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    s = valid_step(); s.hidden = None
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    s = valid_step(); s.fixed_budget = 5; s.cap_T = 10
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    assert "fixed budget" in binding.last_error()
    s = valid_step(); s.cost_c = float("nan")
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    s = valid_step(); s.hidden = FAKE + 8
    assert f(ctypes.byref(s), None) == binding.DSPARK_EALIGN
    s = valid_step(d=4)  # 8 bytes per bf16 row
    assert f(ctypes.byref(s), None) == binding.DSPARK_EALIGN
    s = valid_step(); s.workspace = None
    assert f(ctypes.byref(s), None) == binding.DSPARK_EWORKSPACE
    s = valid_step(); s.workspace_bytes -= 256
    assert f(ctypes.byref(s), None) == binding.DSPARK_EWORKSPACE
    s = valid_step(); s.workspace = FAKE + 16
    assert f(ctypes.byref(s), None) == binding.DSPARK_EWORKSPACE


@pytest.mark.parametrize("field", ["draft_tokens", "packed_ids", "packed_pos", "row_req", "row_k"])
@pytest.mark.parametrize("fixed", [False, True])
def test_score_compact_needs_the_packing_buffers(lib, field, fixed):
    s = valid_step()
    if fixed:
        s.fixed_budget = 3
    setattr(s, field, None)
    assert lib.dspark_score_compact(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    assert field in binding.last_error() and "dspark_score_compact" in binding.last_error()
    # the unfused call does not read them
    if field != "draft_tokens":
        s2 = valid_step()
        setattr(s2, field, None)
        s2.workspace = None  # stops before any launch
        assert lib.dspark_score_budget(ctypes.byref(s2), None) == binding.DSPARK_EWORKSPACE


def test_compact_validation(lib):
    for field in ("L", "row_off", "draft_tokens", "packed_ids", "packed_pos", "row_req", "row_k"):
        s = valid_step()
        setattr(s, field, None)
        assert lib.dspark_compact(ctypes.byref(s), None) == binding.DSPARK_EINVAL, field


def test_verify_validation(lib):
    f = lib.dspark_verify
    for field in ("draft_tokens", "target_logits", "draft_logits", "L", "draft_off", "row_off",
                  "row_req", "row_k", "accept_len", "num_emitted", "out_tokens", "p_tok", "q_tok"):
        s = valid_step()
        setattr(s, field, None)
        assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL, field
    s = valid_step(); s.temperature = -1.0
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    s = valid_step(); s.temperature = float("inf")
    assert f(ctypes.byref(s), None) == binding.DSPARK_EINVAL
    s = valid_step(V=1001)  # bf16 row of 2002 bytes
    assert f(ctypes.byref(s), None) == binding.DSPARK_EALIGN
    s = valid_step(); s.target_logits = FAKE + 4
    assert f(ctypes.byref(s), None) == binding.DSPARK_EALIGN
    s = valid_step(); s.workspace_bytes = 16
    assert f(ctypes.byref(s), None) == binding.DSPARK_EWORKSPACE


def test_version(lib):
    assert "sm_103a" in binding.version()


def test_noalloc_scratch_holds_the_documented_shape(lib):
    """The fixed scratch of dspark_verify_noalloc (less its 256-byte shape
    record) holds the workspace of B=512, gamma=16, V=151936, as the header
    states, and not that of B=1024."""
    room = binding.DSPARK_NOALLOC_SCRATCH_BYTES - 256
    assert binding.dspark_workspace_size(512, 16, 151936, 4096) <= room
    assert binding.dspark_workspace_size(1024, 16, 151936, 4096) > room


def test_wait_bound_setter(lib):
    """The bound of the device waits is a host value read at each launch: set,
    read back, and 0 restores the 2 s default (no GPU needed)."""
    default = binding.dspark_wait_timeout_ns()
    assert default == 2_000_000_000
    try:
        assert binding.dspark_set_wait_timeout_ns(12345) == binding.DSPARK_OK
        assert binding.dspark_wait_timeout_ns() == 12345
    finally:
        binding.dspark_set_wait_timeout_ns(0)
    assert binding.dspark_wait_timeout_ns() == default


def test_cap_accept_needs_a_window(lib):
    s = valid_step()
    assert lib.dspark_verify_cap_accept(ctypes.byref(s), None, None, None, None) == binding.DSPARK_EINVAL
    assert "commit_len" in binding.last_error()
    assert lib.dspark_verify_cap_accept(None, None, None, None, None) == binding.DSPARK_EINVAL


def test_score_entropy_host_checks(lib):
    f = lib.dspark_score_entropy
    f.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]
    assert f(None, 1.0, None) == binding.DSPARK_EINVAL
    s = valid_step()
    for theta in (0.0, -1.0, float("inf"), float("nan")):
        assert f(ctypes.byref(s), theta, None) == binding.DSPARK_EINVAL, theta
        assert "theta" in binding.last_error()
    s.fixed_budget = 3
    assert f(ctypes.byref(s), 1.0, None) == binding.DSPARK_EINVAL
    s = valid_step()
    s.draft_logits = None
    assert f(ctypes.byref(s), 1.0, None) == binding.DSPARK_EINVAL
    assert "draft_logits" in binding.last_error()
    s = valid_step()
    s.draft_logits = FAKE + 8
    assert f(ctypes.byref(s), 1.0, None) == binding.DSPARK_EALIGN


def test_fit_sts_tau_host_checks(lib):
    f = lib.dspark_fit_sts_tau
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P, P, ctypes.c_float, ctypes.c_float,
                  P, P, P, P]
    ok = dict(N=4, gamma=3, conf=FAKE, tu=FAKE, L=FAKE, a=FAKE, lo=0.05, hi=20.0, out=FAKE)

    def call(**kw):
        k = dict(ok, **kw)
        return f(k["N"], k["gamma"], k["conf"], k["tu"], k["L"], k["a"], k["lo"], k["hi"],
                 k["out"], None, None, None)

    for bad in (dict(N=-1), dict(gamma=0), dict(gamma=65), dict(lo=0.0), dict(lo=2.0, hi=1.0),
                dict(hi=float("inf")), dict(lo=float("nan")), dict(tu=None), dict(out=None),
                dict(conf=None), dict(L=None), dict(a=None)):
        assert call(**bad) == binding.DSPARK_EINVAL, bad


def test_binding_checks_variant_arrays_before_the_call():
    """The binding refuses host, mistyped or missized arrays for the variant
    calls before anything reaches the library (no GPU needed)."""
    import torch
    s = binding.DsparkStep()
    s.B = 4
    with pytest.raises(ValueError, match="commit_len must be int32"):
        binding.dspark_verify_cap_accept(s, torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA device memory"):
        binding.dspark_verify_cap_accept(s, torch.zeros(4, dtype=torch.int32))
    with pytest.raises(ValueError, match="required"):
        binding.dspark_verify_cap_accept(s, None)
    conf = torch.zeros((3, 5), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA device memory"):
        binding.dspark_fit_sts_tau(conf, torch.ones(5), torch.zeros(3, dtype=torch.int32),
                                   torch.zeros(3, dtype=torch.int32), torch.zeros(5))
    empty = torch.zeros((0, 5), dtype=torch.float32)   # N = 0: only tau arrays matter
    with pytest.raises(ValueError, match="tau_used must be float32"):
        binding.dspark_fit_sts_tau(empty, torch.ones(5, dtype=torch.float64), None, None,
                                   torch.zeros(5))
    with pytest.raises(ValueError, match="conf must be a"):
        binding.dspark_fit_sts_tau(torch.zeros(5), torch.ones(5), None, None, torch.zeros(5))


def test_a_c_program_builds_against_the_header_and_library(lib):
    """A plain C11 program (warnings as errors) includes dspark.h, links
    libdspark.so and calls the host-side entry points: the ABI needs no C++
    and no Python."""
    src = r'''
#include <stdio.h>
#include "dspark.h"
int main(void) {
    dspark_step s = {0};
    printf("%s\n", dspark_version());
    printf("%zu\n", dspark_workspace_size(256, 16, 129280, 7168));
    printf("%d\n", (int)dspark_verify(NULL, NULL));
    printf("%d\n", (int)dspark_score_entropy(NULL, 1.0f, NULL));
    printf("%d\n", (int)dspark_verify_cap_accept(&s, NULL, NULL, NULL, NULL));
    printf("%d\n", (int)dspark_fit_sts_tau(-1, 4, NULL, NULL, NULL, NULL, 0.1f, 10.0f,
                                           NULL, NULL, NULL, NULL));
    printf("%s\n", dspark_last_error());
    return 0;
}
'''
    libdir = os.path.dirname(binding.lib_path())
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "use.c")
        exe = os.path.join(td, "use")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), c, "-o", exe, "-L", libdir, "-ldspark",
                        f"-Wl,-rpath,{libdir}"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0] == binding.version()
    assert int(out[1]) == binding.dspark_workspace_size(256, 16, 129280, 7168)
    # B = 0 in a zeroed struct: check_shape rejects gamma = 0 first
    assert [int(x) for x in out[2:6]] == [binding.DSPARK_EINVAL] * 4
    assert "N=-1" in out[6]
