"""The C-ABI library loads and exports every symbol include/jt.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import re
import os


import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    hdr = open(os.path.join(ROOT, "include", "jt.h")).read()
    return set(re.findall(r"^\s*(?:jt_status|size_t|const char\*|int)\s+(jt_\w+)\s*\(", hdr, re.M))


def test_library_exports_every_declared_symbol():
    lib = jt.load()
    declared = _declared()
    assert declared == set(binding.EXPORTS)
    raw = ctypes.CDLL(jt.library_path())
    for name in declared:
        assert hasattr(raw, name), name


def test_status_strings_and_version():
    for code in (0, -1, -2, -3, -4, -5):
        assert jt.jt_status_str(code).startswith("JT_")
    assert jt.jt_version() >= 10000


def test_host_side_checks_need_no_gpu():
    lib = jt.load()
    P = ctypes.c_void_p
    # null pointers / bad sizes are rejected before anything is enqueued
    assert lib.jt_tree_build(None, None, None, 1, 4, 2, 10, 1, None, None, None, None, None, 0, None) == -1
    assert lib.jt_tree_attn_paged(None, None, None, 1, None, 1, 1, None, None, None, 1, 1, 1, 32, 8,
                                  128, 16, 0.1, None, None, None, 0, None) == -1
    assert lib.jt_verify_accept(None, None, None, None, 1, 4, 10, 1, 0, 0.0, None, None, None, None,
                                0, None) == -1
    assert lib.jt_tree_topw(None, 1, 10, 2, None, None, None, None, 0, None) == -1
    # workspace sizes are pure host arithmetic for the build and accept ops
    assert jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, 8, 16, 4, 151936) > 0
    assert jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, 8, 16, 9, 151936) == 0
    assert jt.jt_workspace_size(jt.JT_OP_VERIFY_ACCEPT, 8, 0, 0, 0, 2048) > 0


def test_checks_variant_builds_and_exports_every_symbol():
    """The debug variant (-DJT_CHECKS device-side input checks, -DJT_NVTX
    ranges) builds for sm_103a and exports the same entry points."""
    from tree_speculative_decoding_jt_gb300 import build as b

    path = b.build(variant="checks")
    assert path.endswith("libjt_checks.so") and os.path.exists(path)
    raw = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(raw, name), name
    # the host-side checks answer the same way in the variant
    raw.jt_tree_topw.restype = ctypes.c_int
    assert raw.jt_tree_topw(None, ctypes.c_int64(1), ctypes.c_int64(10), 2, None, None, None, None,
                            ctypes.c_size_t(0), None) == -1


def test_package_exports_the_status_codes():
    """The package root re-exports the jt_status codes of include/jt.h
    (JtError.status is compared with them)."""
    import tree_speculative_decoding_jt_gb300 as jt
    assert (jt.JT_OK, jt.JT_ERR_INVALID, jt.JT_ERR_UNSUPPORTED, jt.JT_ERR_CUDA, jt.JT_ERR_TIMEOUT,
            jt.JT_ERR_WORKSPACE) == (0, -1, -2, -3, -4, -5)
    hdr = open(os.path.join(ROOT, "include", "jt.h")).read()
    for name, val in (("JT_ERR_INVALID", -1), ("JT_ERR_UNSUPPORTED", -2), ("JT_ERR_CUDA", -3),
                      ("JT_ERR_TIMEOUT", -4), ("JT_ERR_WORKSPACE", -5)):
        assert f"{name} = {val}" in hdr
