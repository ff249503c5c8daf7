"""Host-side checks of the timeout diagnostic entry point (no device work):
a missing, misaligned or too small workspace is refused before any launch."""
import ctypes

import tree_speculative_decoding_jt_gb300 as jt

JT_ERR_WORKSPACE = -5


def test_bad_workspace_is_refused():
    lib = jt.load()
    assert lib.jt_selftest_wait_timeout(None, 256, None) == JT_ERR_WORKSPACE
    assert lib.jt_selftest_wait_timeout(ctypes.c_void_p(4096 + 8), 256, None) == JT_ERR_WORKSPACE
    assert lib.jt_selftest_wait_timeout(ctypes.c_void_p(4096), 128, None) == JT_ERR_WORKSPACE
