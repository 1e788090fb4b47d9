"""The C-ABI library builds, loads and exports every declared symbol (CPU only).

Also checks the host-side argument validation, which runs before any CUDA
call and therefore needs no GPU.
"""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

RC_OK, RC_ERR_INVALID = 0, 1


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from ring_collectives_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    for want in ("ring_ppermute_right", "ring_all_gather", "ring_reduce_scatter", "ring_allreduce", "ag_gemm",
                 "ring_status", "ring_last_error", "ring_set_timeout_ms"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _call(lib, name, *args):
    f = getattr(lib, name)
    f.restype = ctypes.c_int
    return f(*args)


def test_validation_rejects_bad_arguments_without_a_gpu(lib):
    vp = ctypes.c_void_p
    sz = ctypes.c_size_t
    fake = vp(0x10000)  # never dereferenced: validation fails first
    lib.ring_last_error.restype = ctypes.c_char_p
    # N not a multiple of P
    assert _call(lib, "ring_allreduce", fake, sz(4096), 4, sz(10), 0, vp(0)) == RC_ERR_INVALID
    assert b"multiple" in lib.ring_last_error()
    # P out of range
    assert _call(lib, "ring_allreduce", fake, sz(4096), 0, sz(8), 0, vp(0)) == RC_ERR_INVALID
    assert _call(lib, "ring_allreduce", fake, sz(4096), 65, sz(65), 0, vp(0)) == RC_ERR_INVALID
    # unknown dtype
    assert _call(lib, "ring_allreduce", fake, sz(4096), 4, sz(8), 7, vp(0)) == RC_ERR_INVALID
    # stride smaller than a slot
    assert _call(lib, "ring_allreduce", fake, sz(16), 4, sz(8), 0, vp(0)) == RC_ERR_INVALID
    # null base
    assert _call(lib, "ring_allreduce", vp(0), sz(4096), 4, sz(8), 0, vp(0)) == RC_ERR_INVALID
    # overlapping ppermute src/dst
    assert _call(lib, "ring_ppermute_right", fake, sz(64), vp(0x10020), sz(64), 4, sz(16), 0, vp(0)) == RC_ERR_INVALID
    # all_gather out stride below P*n
    assert _call(lib, "ring_all_gather", fake, sz(64), vp(0x20000), sz(64), 4, sz(16), 0, vp(0)) == RC_ERR_INVALID
    # reduce_scatter out overlapping bufs
    assert _call(lib, "ring_reduce_scatter", fake, sz(4096), vp(0x10010), sz(64), 4, sz(16), 0, vp(0)) == RC_ERR_INVALID
    # fault-injection hooks: bad arguments are refused, -1 cancels
    assert _call(lib, "ag_gemm_debug_skip_piece", -2) == RC_ERR_INVALID
    assert _call(lib, "ag_gemm_debug_skip_piece", -1) == 0
    assert _call(lib, "ring_debug_skip_notify", -2, 0) == RC_ERR_INVALID
    assert _call(lib, "ring_debug_skip_notify", -1, -1) == 0
    # timeout bounds
    assert _call(lib, "ring_set_timeout_ms", ctypes.c_uint(0)) == RC_ERR_INVALID


def test_degenerate_sizes_are_no_ops_without_a_gpu(lib):
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    assert _call(lib, "ring_allreduce", vp(0), sz(0), 4, sz(0), 0, vp(0)) == RC_OK
    assert _call(lib, "ring_allreduce", vp(0x10000), sz(0), 1, sz(8), 0, vp(0)) == RC_OK
    assert _call(lib, "ring_all_gather", vp(0), sz(0), vp(0), sz(0), 4, sz(0), 0, vp(0)) == RC_OK


def test_python_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import ring_collectives_gb300 as rc
    monkeypatch.setattr(rc, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rc, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        rc.load()


def test_binding_declares_every_header_function_with_its_result_type():
    """The ctypes table covers every function of include/ringcoll.h, with the
    header's result type (size_t, const char *, or int)."""
    import ctypes
    import re
    import ring_collectives_gb300 as rc
    with open(os.path.join(ROOT, "include", "ringcoll.h"), encoding="utf-8") as f:
        text = f.read()
    decls = dict((name, ret.strip()) for ret, name in
                 re.findall(r"^(int|size_t|const char \*)\s*(\w+)\(", text, flags=re.M))
    assert set(decls) == set(rc._SIGNATURES), set(decls) ^ set(rc._SIGNATURES)
    want = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char *": ctypes.c_char_p}
    L = rc.load()
    for name, ret in decls.items():
        assert getattr(L, name).restype is want[ret], name


def test_ex_variants_validate_and_size_without_a_gpu(lib):
    """The caller-workspace variants reject a null workspace before any CUDA
    call; the GEMM sizing functions need no device."""
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    fake = vp(0x10000)
    assert _call(lib, "ring_reduce_scatter_ex", fake, sz(4096), vp(0x20000), sz(1024), 4, sz(16), 0, vp(0), sz(0),
                 vp(0)) == RC_ERR_INVALID
    assert _call(lib, "ring_all_gather_ex", fake, sz(64), vp(0x20000), sz(256), 4, sz(16), 0, vp(0), sz(0),
                 vp(0)) == RC_ERR_INVALID
    assert _call(lib, "ring_status_ex", vp(0), vp(0)) == RC_ERR_INVALID
    assert _call(lib, "ring_status_ex", vp(0x10004), vp(0)) == RC_ERR_INVALID   # not 16-byte aligned
    lib.ag_gemm_workspace_bytes.restype = ctypes.c_size_t
    lib.gemm_rs_workspace_bytes.restype = ctypes.c_size_t
    assert lib.ag_gemm_workspace_bytes(8, 1024) == 128 + 4 * 8 * 1024 // 16
    assert lib.ag_gemm_workspace_bytes(8, 100) == 0
    assert lib.gemm_rs_workspace_bytes(8, 8192, 4096, 512) == 128
