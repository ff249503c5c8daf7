"""Host-side argument handling of jt_tree_build_mixed (no device work): an
alpha outside [0, 1] is refused before any CUDA call, and the mixed build's
workspace holds the plain build's plus the entropy partials."""
import ctypes

import tree_speculative_decoding_jt_gb300 as jt

JT_ERR_INVALID = -1


def test_alpha_outside_range_is_refused_on_the_host():
    lib = jt.load()
    fake = ctypes.c_void_p(4096)          # never dereferenced: refused before any CUDA call
    for alpha in (1.0 + 2 ** -52, 1.5, -1e-300, float("nan"), float("inf")):
        rc = lib.jt_tree_build_mixed(fake, fake, fake, 2, 3, 2, 100, 10, alpha, fake, fake, fake, fake,
                                     fake, 1 << 20, None)
        assert rc == JT_ERR_INVALID, alpha


def test_mixed_workspace_is_larger_than_the_plain_one():
    for nseq, N, W, V in ((1, 1, 1, 5), (8, 16, 4, 151936), (64, 8, 8, 32000)):
        plain = jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, nseq, N, W, V)
        mixed = jt.jt_workspace_size(jt.JT_OP_TREE_BUILD_MIXED, nseq, N, W, V)
        assert plain > 0 and mixed > plain
    assert jt.jt_workspace_size(jt.JT_OP_TREE_BUILD_MIXED, 1, 1, 9, 100) == 0   # W > 8
