"""The kernels' failure path, without a GPU fault: a bounded mbarrier wait that runs out sets the
library's device error flag and the kernel returns, leaving the context usable.  The self-test
launch waits on a barrier that nothing arrives on, with the same bounded wait and flag as the
verify and prompt pipelines."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_sets_the_flag_and_the_context_stays_usable(lib):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8, kvq8_device_error, kvq8_selftest_wait_timeout
    assert kvq8_device_error(reset=True) in (0, 1)
    assert kvq8_device_error(reset=False) == 0            # cleared
    kvq8_selftest_wait_timeout(4096)
    torch.cuda.synchronize()
    assert kvq8_device_error(reset=False) == 1            # the wait gave up and said so
    assert kvq8_device_error(reset=True) == 1             # read, then cleared
    assert kvq8_device_error(reset=False) == 0
    # the context still works: a verify call right after matches the oracle, with the flag clear
    inp = workloads.random_small(5, 6, 1, 256, 700, 4)
    gpu, orc = build_caches(inp)
    out = attn_verify_q8(torch.from_numpy(np.ascontiguousarray(inp.q, np.float32)).cuda(), gpu, 700, 696, 1.0 / 16.0)
    torch.cuda.synchronize()
    ref = oracle.attention(orc, inp.q, 700, 696, 1.0 / 16.0)
    assert rel_err(out.cpu().numpy(), ref) <= VERIFY_TOL
    assert kvq8_device_error(reset=True) == 0


def test_wait_timeout_rejects_bad_poll_counts(lib):
    from speculative_verify_attention_gb300 import KVQ8Error, kvq8_selftest_wait_timeout
    for polls in (0, -1, (1 << 20) + 1):
        with pytest.raises(KVQ8Error):
            kvq8_selftest_wait_timeout(polls)
