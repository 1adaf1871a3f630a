"""Failure detection without a GPU fault: a kernel's bounded wait that runs out records
LA_ERR_TIMEOUT in the device status word and returns; the context stays usable."""
import pytest

import compressive_memory_attention_02_b300 as la


def test_selftest_rejects_bad_limits_on_host():
    assert la.lib.la_selftest_wait_timeout(0, None) == la.LA_ERR_INVALID_ARG
    assert la.lib.la_selftest_wait_timeout((1 << 32) + 1, None) == la.LA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_wait_that_runs_out_reports_timeout_and_context_survives():
    import numpy as np
    import torch

    import oracle
    import synthetic
    from gpu_helpers import TOL_BF16, fwd, to_dev, to_host

    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    la.la_selftest_wait_timeout(2_000_000)          # about 1 ms at the SM clock
    assert la.la_get_last_device_status() == la.LA_ERR_TIMEOUT
    assert la.la_get_last_device_status() == la.LA_OK   # reading clears the word
    # the device still computes correctly afterwards
    q = synthetic.normal(71, 0, (1, 2, 300, 128), 0.5, "bf16")
    k = synthetic.normal(71, 1, (1, 2, 300, 128), 0.5, "bf16")
    v = synthetic.normal(71, 2, (1, 2, 300, 128), 0.5, "bf16")
    out, M, z = fwd(to_dev(q), to_dev(k), to_dev(v))
    r_out, _, _ = oracle.causal_fwd(q, k, v)
    assert oracle.rel_err_rows(to_host(out), r_out) <= TOL_BF16
