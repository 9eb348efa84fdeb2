"""CPU-side checks of the C ABI: the library builds, loads, and exports every
entry point include/rcu.h declares; the Python binding's host logic
(canonical strides) behaves.  No compute call runs here (no GPU)."""
import ctypes
import os
import re

import pytest
import torch

from recurrent_cell_unroll_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    return ctypes.CDLL(path)


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "rcu.h")).read()
    return sorted(set(re.findall(r"^RCU_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("rnn_create", "rnn_set_weights", "rnn_forward", "rssm_unroll"):
        assert required in names
    assert set(names) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"librcu.so does not export {name}"


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {n for n in exported if n.startswith(("rnn_", "rssm_", "rcu_"))}
    assert ours == set(declared_symbols())


def test_version_string_without_gpu(lib):
    lib.rcu_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.rcu_version()


def test_canonical_contiguous():
    base = torch.arange(20, dtype=torch.float32)
    t = base.as_strided((1, 4, 5), (5, 5, 1))
    assert t.is_contiguous()
    c = binding.canonical_contiguous(t)
    assert c.stride() == (20, 5, 1) and torch.equal(c, t)
    u = torch.zeros(2, 3, 4)
    assert binding.canonical_contiguous(u) is u
    v = torch.zeros(4, 3).t()
    assert binding.canonical_contiguous(v).stride() == (4, 1)


def test_binding_rejects_host_tensors():
    with pytest.raises(ValueError):
        binding._dev(torch.zeros(3))


def test_binding_checks_tensor_shapes_before_the_call():
    """The C ABI reads each buffer at the size (T, B) and the handle imply, so
    the wrapper refuses a tensor of any other shape (a bidirectional net
    wants dy [T, B, 2*Hout])."""
    from types import SimpleNamespace
    net = SimpleNamespace(in_dim=16, layers=2, D=2, Hout=32, hidden=32)
    x = torch.zeros(5, 3, 16)
    ok = dict(lengths=torch.zeros(3), h0=torch.zeros(4, 3, 32), c0=torch.zeros(4, 3, 32))
    assert binding.RNN._shapes(net, x, **ok, dy=torch.zeros(5, 3, 64),
                               dh_n=torch.zeros(4, 3, 32)) == (5, 3)
    bad = [dict(dy=torch.zeros(5, 3, 32)), dict(h0=torch.zeros(2, 3, 32)),
           dict(lengths=torch.zeros(4)), dict(out=torch.zeros(5, 3, 63)),
           dict(dc_n=torch.zeros(4, 2, 32))]
    for kw in bad:
        with pytest.raises(ValueError):
            binding.RNN._shapes(net, x, **kw)
    with pytest.raises(ValueError):
        binding.RNN._shapes(net, torch.zeros(5, 3, 15))


def test_constants_match_header():
    """Every RCU_* value the binding names is the header's #define."""
    import re
    text = open(os.path.join(ROOT, "include", "rcu.h")).read()
    defs = {m.group(1): int(m.group(2), 0) for m in
            re.finditer(r"#define\s+(RCU_\w+)\s+\(?(-?(?:0x[0-9a-fA-F]+|\d+))\)?", text)}
    named = [n for n in dir(binding) if n.startswith("RCU_")]
    assert len(named) >= 10
    for n in named:
        assert n in defs, f"{n} is not defined in rcu.h"
        assert getattr(binding, n) == defs[n], n



def _declarations():
    """{name: (return type, [parameter declarations])} of every RCU_API function."""
    src = open(os.path.join(ROOT, "include", "rcu.h")).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    out = {}
    for m in re.finditer(r"RCU_API\s+([\w\s\*]*?)\b(\w+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(3).split(",")]
        if params == ["void"] or params == [""]:
            params = []
        out[m.group(2)] = (" ".join(m.group(1).split()), params)
    return out


def _kind_of_c(decl: str) -> str:
    decl = " ".join(decl.split())
    if "*" in decl or decl.startswith(("rcu_rnn_t", "rcu_rssm_t")):
        return "ptr"
    if decl.startswith("int64_t"):
        return "i64"
    if decl.startswith("double"):
        return "f64"
    if decl.startswith("float"):
        return "f32"
    if decl.startswith("int"):
        return "i32"
    raise AssertionError(f"unclassified parameter {decl!r}")


def _kind_of_ctypes(t) -> str:
    if t in (ctypes.c_void_p, ctypes.c_char_p) or isinstance(t, type(ctypes.POINTER(ctypes.c_int))):
        return "ptr"
    return {ctypes.c_int: "i32", ctypes.c_int64: "i64", ctypes.c_double: "f64",
            ctypes.c_float: "f32"}[t]


def test_binding_signatures_match_the_header():
    """Every declared entry point has ctypes argtypes (without them a pointer
    argument would be passed as a C int), with the header's parameter count
    and kinds, and a matching return type."""
    decls = _declarations()
    sigs = binding.signatures()
    assert set(decls) == set(sigs)
    for name, (ret, params) in decls.items():
        res, args = sigs[name]
        want = [_kind_of_c(p) for p in params]
        got = [_kind_of_ctypes(a) for a in args]
        assert got == want, f"{name}: binding {got} vs header {want}"
        assert (res is ctypes.c_char_p) == ("char" in ret), name
        if "char" not in ret:
            assert res is ctypes.c_int and ret == "int", name


def test_null_handle_errors_reach_rcu_last_error(lib):
    """Argument errors from both halves of the host code (stacked networks,
    RSSM) return RCU_ERR_INVALID and leave their message for rcu_last_error on
    this thread; a NULL handle is checked before any CUDA call, so this runs
    without a GPU."""
    sigs = binding.signatures()
    for name in ("rnn_get_weight_grads", "rnn_set_attr", "rnn_profile_entry",
                 "rssm_get_weight_grads", "rssm_get_actor_grads", "rssm_set_attr",
                 "rssm_profile_entry", "rssm_backward", "rssm_backward_actor"):
        fn = getattr(lib, name)
        res, args = sigs[name]
        fn.restype, fn.argtypes = res, args
        zeros = [None if a is not ctypes.c_int and a is not ctypes.c_int64 else 0 for a in args]
        rc = fn(*zeros)
        assert rc == binding.RCU_ERR_INVALID, (name, rc)
        lib.rcu_last_error.restype = ctypes.c_char_p
        msg = lib.rcu_last_error().decode()
        assert name.split("_", 1)[0] in msg and "NULL handle" in msg, (name, msg)


def test_debug_build_compiles_and_exports_the_same_symbols():
    """The RCU_DEBUG build (device bounds checks recorded as an error code
    instead of a faulting access) compiles and exports the same entry points."""
    import subprocess
    path = _build.build(debug=True)
    assert path.endswith("librcu_debug.so") and os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert {n for n in exported if n.startswith(("rnn_", "rssm_", "rcu_"))} == \
        set(declared_symbols())
