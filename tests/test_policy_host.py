"""Host-side argument handling of jt_tree_policy and jt_tree_build_adaptive
(no device work): parameters outside their ranges and a capacity below
nseq x the policy's ceiling are refused before any CUDA call."""
import ctypes

import tree_speculative_decoding_jt_gb300 as jt

JT_ERR_INVALID = -1
FAKE = ctypes.c_void_p(4096)   # never dereferenced: refused before any CUDA call


def _policy(prm, nseq=4, N=6, W=3):
    return jt.load().jt_tree_policy(FAKE, nseq, N, W, None, ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, 256, None)


def test_bad_policy_parameters_are_refused():
    bad = [dict(b_min=0), dict(b_max=257), dict(b_min=20, b_max=10), dict(w_min=0), dict(w_min=4),
           dict(n_min=7), dict(n_min=-1), dict(n_slack=7), dict(n_slack=-1), dict(beta=0.0), dict(beta=1.01),
           dict(node_cap=-5), dict(log_conf=float("nan")), dict(acc_thresh=float("nan"))]
    for kw in bad:
        assert _policy(jt.policy_params(**kw)) == JT_ERR_INVALID, kw
    lib = jt.load()
    assert lib.jt_tree_policy(FAKE, 4, 0, 3, None, ctypes.byref(jt.policy_params()), FAKE, FAKE, FAKE, FAKE,
                              FAKE, FAKE, 256, None) == JT_ERR_INVALID       # N = 0


def test_adaptive_build_capacity_must_cover_the_ceiling():
    lib = jt.load()
    prm = jt.policy_params(b_min=8, b_max=64, node_cap=100)     # ceiling min(64, max(8, 100 // 4)) = 25
    assert jt.policy_ceiling(prm, 4) == 25
    for cap in (0, 99):
        rc = lib.jt_tree_build_adaptive(FAKE, FAKE, 4, 6, 3, 1000, cap, None, ctypes.byref(prm), FAKE, FAKE,
                                        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
        assert rc == JT_ERR_INVALID, cap
    assert jt.policy_ceiling(jt.policy_params(b_min=30, node_cap=100), 4) == 30
    assert jt.policy_ceiling(jt.policy_params(b_max=200), 4) == 200


def test_policy_workspace_is_the_header():
    assert jt.jt_workspace_size(jt.JT_OP_TREE_POLICY) == 256
