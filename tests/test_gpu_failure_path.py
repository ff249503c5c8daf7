"""The device-side failure path without a GPU fault: a bounded wait that
nothing completes runs out (the library's 2 s limit), the kernel raises the
timeout flag and exits, the host reads JT_ERR_TIMEOUT from the workspace,
and the CUDA context stays usable (a later call computes the right
result)."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from gpu_util import dev

pytestmark = pytest.mark.gpu

JT_ERR_TIMEOUT = -4


def test_wait_that_nothing_completes_reports_timeout_and_context_survives():
    ws = jt.jt_selftest_wait_timeout()
    with pytest.raises(jt.JtError) as e:
        jt.jt_check(ws)
    assert e.value.status == JT_ERR_TIMEOUT
    jt.jt_check(ws)  # jt_check cleared the flag
    # the context is still usable: a top-W call gives the oracle's ids
    rng = np.random.default_rng(3)
    z = (rng.standard_normal((3, 5000)) * np.sqrt(2)).astype(np.float32)
    tok, lp, lse = jt.jt_tree_topw(dev(z), 4)
    torch.cuda.synchronize()
    otok, _, olse = oracle.topw_lse(z, 4)
    np.testing.assert_array_equal(tok.cpu().numpy(), otok)
    assert np.abs(lse.cpu().numpy() - olse).max() <= 1e-9
