"""Host-only checks of the C-ABI library: it loads without a GPU, exports every
function ``include/mhcpb.h`` declares, and rejects bad flags and shapes before
making any CUDA call (the cuDNN frontend page "DSv4.1 mHC projection/RMS
backward", "Requirements and tensor contract": other shapes and precisions are
rejected; allow_tf32 must be passed explicitly)."""
import ctypes
import os
import re

import pytest

from rms_backward_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mhcpb.h")


def _built():
    return os.path.exists(abi.LIB_PATH)


@pytest.fixture(scope="module")
def lib():
    if not _built():
        from rms_backward_gb300 import build
        try:
            build.build()
        except RuntimeError as e:  # pragma: no cover
            pytest.skip(f"cannot build libmhcpb.so here: {e}")
    return abi.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(mhcpb_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mhcpb_plan_create", "mhcpb_workspace_bytes", "mhcpb_execute", "mhcpb_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(abi.EXPORTED) <= set(declared_functions())


def test_status_strings(lib):
    for s in range(0, 11):
        assert abi.status_string(s)
    assert abi.status_string(12345) == "unknown status"


@pytest.mark.parametrize("T,K,flags,status", [
    (100, 512, 0, abi.MHCPB_ERR_TF32_NOT_ALLOWED),
    (100, 512, abi.MHCPB_HAS_ADDEND, abi.MHCPB_ERR_TF32_NOT_ALLOWED),
    (100, 512, abi.MHCPB_ALLOW_TF32 | 64, abi.MHCPB_ERR_INVALID_ARG),
    (-1, 512, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    (-5, 512, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    (100, 0, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    (100, 12, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    (100, 4, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    ((1 << 24) + 1, 512, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
    (100, (1 << 20) + 8, abi.MHCPB_ALLOW_TF32, abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
])
def test_plan_create_rejects_before_cuda(lib, T, K, flags, status):
    with pytest.raises(abi.MhcpbError) as ei:
        abi.mhcpb_plan_create(T, K, 0, flags)
    assert ei.value.status == status


def test_empty_batch_passes_the_shape_check(lib):
    """T = 0 is a valid shape (an empty batch: dW = 0).  Without a GPU the
    call then fails at the device query, not at the shape check."""
    try:
        h = abi.mhcpb_plan_create(0, 512, 0, abi.MHCPB_ALLOW_TF32)
    except abi.MhcpbError as e:
        assert e.status != abi.MHCPB_ERR_UNSUPPORTED_SHAPE
    else:   # on a GPU machine the plan is created
        assert abi.mhcpb_workspace_bytes(h) == 0
        abi.mhcpb_destroy(h)


def test_null_arguments_rejected(lib):
    import ctypes
    assert lib.mhcpb_plan_create(None, 10, 16, 0, 1) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_workspace_bytes(None, None) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_execute(None, *([None] * 8), 0, None, None) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_execute_dx(None, *([None] * 7), 0, None, None) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_reduce_dw(None, None, 0, None, None) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_plan_query(None, 0, None) == abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_destroy(None) == abi.MHCPB_OK
    v = ctypes.c_int()
    assert lib.mhcpb_get_device_status(None, ctypes.byref(v), 0) == abi.MHCPB_ERR_INVALID_ARG


def test_workspace_formula_matches_page_size():
    # S * 24 * K * 4 with S = ceil(T / 512): 15,728,640 bytes at T=4096, K=20480,
    # the workspace size the page states for the training profile.
    T, K = 4096, 20480
    S = -(-T // abi.MHCPB_PARTIAL_TOKENS(T))
    assert S * 24 * K * 4 == 15_728_640


def test_missing_library_fails_loudly():
    """No CPU fallback: without the built library the binding raises (run in a
    fresh interpreter so the already loaded library is not reused)."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from rms_backward_gb300 import abi\n"
            "try:\n"
            "    abi.load('/nonexistent/libmhcpb.so')\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'missing' in str(e))\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert out.stdout.strip() == "raised True", out.stdout + out.stderr


_SCALARS = {"int64_t": ctypes.c_int64, "uint64_t": ctypes.c_uint64, "int": ctypes.c_int,
            "uint32_t": ctypes.c_uint32, "size_t": ctypes.c_size_t, "float": ctypes.c_float,
            "mhcpb_status_t": ctypes.c_int}
_POINTERS = ("mhcpb_plan_t",)   # typedef of a struct pointer


def declared_signatures():
    """(return type, [parameter types]) of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    out = {}
    for ret, name, params in re.findall(
            r"(mhcpb_status_t|const\s+char\s*\*)\s*(mhcpb_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        types = []
        for p in (q.strip() for q in params.split(",")):
            if p in ("", "void"):
                continue
            types.append(re.sub(r"\s*\b[A-Za-z_][A-Za-z0-9_]*$", "", p).strip())   # drop the name
        out[name] = (ret.replace(" ", ""), types)
    return out


def _same_kind(c_type, ct):
    if "*" in c_type or c_type in _POINTERS:
        return ct is ctypes.c_void_p or issubclass(ct, ctypes._Pointer)
    base = _SCALARS[c_type.replace("const ", "")]
    return ctypes.sizeof(ct) == ctypes.sizeof(base) and (ct is base or ct._type_ == base._type_)


def test_binding_signatures_match_the_header(lib):
    """The ctypes declarations agree with the C prototypes: the same number of
    arguments and, position by position, the same size and pointer-ness (a
    mismatch would pass garbage through the ABI without any error)."""
    sigs = declared_signatures()
    assert set(sigs) == set(declared_functions())
    for name, (ret, types) in sigs.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == len(types), (name, types, fn.argtypes)
        for i, (c_type, ct) in enumerate(zip(types, fn.argtypes)):
            assert _same_kind(c_type, ct), (name, i, c_type, ct)
        if ret == "mhcpb_status_t":
            assert fn.restype in (ctypes.c_int, ctypes.c_int32), name
        else:
            assert fn.restype is ctypes.c_char_p, name


def _header_constants():
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    consts = {}
    for name, expr in re.findall(r"\b(MHCPB_[A-Z0-9_]+)\s*=\s*([^,}\n]+)", text):
        consts[name] = expr
    for name, expr in re.findall(r"#define\s+(MHCPB_[A-Z0-9_]+)\s+(\([^)\n]*\)|[0-9][^\s]*)", text):
        consts[name] = expr
    out = {}
    for name, expr in consts.items():
        py = re.sub(r"(\d)u\b", r"\1", expr.strip())
        if re.fullmatch(r"[0-9()<\s+*-]+", py):
            out[name] = eval(py)   # integer literals and shifts only (checked above)
    return out


def test_binding_constants_match_the_header():
    consts = _header_constants()
    for name in ("MHCPB_OK", "MHCPB_ERR_SCRATCH_TOO_SMALL", "MHCPB_ALLOW_TF32",
                 "MHCPB_TEST_INJECT_STALL", "MHCPB_STATIC_SCRATCH_BYTES", "MHCPB_NPROJ"):
        assert name in consts, name           # the parser sees both forms
    checked = 0
    for name, value in consts.items():
        if hasattr(abi, name) and not callable(getattr(abi, name)):
            assert getattr(abi, name) == value, name
            checked += 1
    assert checked >= 20
    # the macro of the partial size: 512 tokens for every T
    m = re.search(r"#define\s+MHCPB_PARTIAL_TOKENS\(T\)\s+(\d+)", open(HEADER).read())
    for T in (1, 512, 4096, 1 << 24):
        assert abi.MHCPB_PARTIAL_TOKENS(T) == int(m.group(1))


def test_checked_sites_in_a_normal_build(lib):
    """A normal build reports itself unchecked with every site 0, without any
    CUDA call (so it works here, with no GPU); NULL arguments are rejected."""
    checked, sites = abi.mhcpb_debug_checked_sites()
    assert checked is False and set(sites.values()) == {0} and len(sites) == 5
    import ctypes
    assert lib.mhcpb_debug_checked_sites(None, None) == abi.MHCPB_ERR_INVALID_ARG
    one = ctypes.c_int()
    assert lib.mhcpb_debug_checked_sites(None, ctypes.byref(one)) == abi.MHCPB_ERR_INVALID_ARG
