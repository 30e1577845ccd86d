"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every entry point
declared in include/lapl_attn.h, and rejects bad configurations before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from conftest import build_library
    build_library()
    from laplacian_nystr_attention_gb300 import _lib
    return _lib


def declared_entry_points():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(lapl_attn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_entry_points()
    for required in ["lapl_attn_create", "lapl_attn_forward", "lapl_attn_destroy",
                     "lapl_attn_workspace_size", "lapl_attn_forward_debug"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"
    assert set(declared_entry_points()) <= set(lib.EXPORTED)


def test_library_does_not_link_the_oracle(lib):
    data = open(lib.LIB_PATH, "rb").read()
    assert b"orc_forward" not in data and b"lapl_oracle" not in data


def test_status_strings(lib):
    assert lib.lapl_attn_status_string(0) == "LAPL_OK"
    assert lib.lapl_attn_status_string(3) == "LAPL_ERR_WORKSPACE"
    assert lib.lapl_attn_status_string(99) == "LAPL_ERR_UNKNOWN"
    assert lib.lapl_attn_version() >= 100


def test_config_struct_matches_header(lib):
    """The ctypes mirror of lapl_attn_config lists the header's fields, in order, all 4 bytes."""
    src = open(os.path.join(ROOT, "include", "lapl_attn.h")).read()
    body = re.search(r"typedef struct \{(.*?)\} lapl_attn_config;", src, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            names += [t.strip().split()[-1] for t in decl.split(",")]
    py = [n if n != "lam" else "lambda" for n, _ in lib.lapl_attn_config._fields_]
    assert py == names
    assert ctypes.sizeof(lib.lapl_attn_config) == 4 * len(names)


def base_cfg(lib, **kw):
    c = dict(batch=1, heads=1, grid_h=16, grid_w=16, head_dim=32, num_landmarks=16, lam=4.0,
             eps=1e-3, delta=1e-5, ns_steps=20, whiten=1, in_dtype=0, out_dtype=0)
    c.update(kw)
    return lib.lapl_attn_config(**c)


@pytest.mark.parametrize("bad,status", [
    (dict(num_landmarks=15), 2),      # not a perfect square
    (dict(num_landmarks=81), 2),      # s = 9 > 8
    (dict(num_landmarks=9), 2),       # 16 % 3 != 0
    (dict(head_dim=12), 2),           # not a multiple of 8
    (dict(head_dim=136), 2),          # > 128
    (dict(lam=0.0), 1),
    (dict(lam=-1.0), 1),
    (dict(eps=-1e-3), 1),
    (dict(delta=0.0), 1),
    (dict(ns_steps=-1), 1),
    (dict(ns_steps=1001), 1),
    (dict(heads=0), 1),
    (dict(batch=-1), 1),
    (dict(in_dtype=7), 1),
    (dict(whiten=2), 1),
    (dict(kernel=2), 1),
    (dict(kernel=-1), 1),
    (dict(solver=2), 1),
    (dict(solver=-1), 1),
])
def test_create_rejects_bad_configs(lib, bad, status):
    h = ctypes.c_void_p()
    st = lib.LIB.lapl_attn_create(ctypes.byref(base_cfg(lib, **bad)), ctypes.byref(h))
    assert st == status
    assert not h.value


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.LIB.lapl_attn_create(None, ctypes.byref(h)) == 1
    assert lib.LIB.lapl_attn_create(ctypes.byref(base_cfg(lib)), None) == 1
    n = ctypes.c_size_t()
    assert lib.LIB.lapl_attn_workspace_size(None, ctypes.byref(n)) == 1
    assert lib.LIB.lapl_attn_forward(None, None, None, None, None, None, None, 0, None) == 1
    assert lib.LIB.lapl_attn_destroy(None) == 0
    assert lib.LIB.lapl_attn_last_error(None) == b""


def test_python_binding_raises_typed_errors(lib):
    with pytest.raises(lib.LaplAttnError) as ei:
        lib.lapl_attn_create(base_cfg(lib, num_landmarks=15))
    assert ei.value.status == lib.LAPL_ERR_UNSUPPORTED


def test_binding_wraps_every_declared_entry_point(lib):
    """The Python binding carries a same-name wrapper for every entry point the header
    declares (argument marshalling only)."""
    for name in declared_entry_points():
        assert callable(getattr(lib, name, None)), name


def test_plan_info_struct_matches_header(lib):
    """The ctypes mirror of lapl_attn_plan_info lists the header's int fields, in order."""
    src = open(os.path.join(ROOT, "include", "lapl_attn.h")).read()
    end = src.index("} lapl_attn_plan_info;")
    body = src[src.rindex("typedef struct {", 0, end):end]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"int\s+(\w+);", body)
    assert names == [n for n, _ in lib.lapl_attn_plan_info._fields_]
