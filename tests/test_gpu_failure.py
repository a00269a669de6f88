"""Failure detection without a GPU fault: every pipeline wait in the kernels is bounded, and a wait
that runs out reports MLA_DEV_WAIT_TIMEOUT through the caller's status word and lets the kernel
return. The self-test waits on a barrier that nothing arrives on; the context must then still run
a decode that matches the oracle."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from parity_util import compare_decode, run_decode

pytestmark = pytest.mark.gpu

MLA_DEV_WAIT_TIMEOUT = 0x4


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    import torch
    import mla_latent_kv_gb300 as mla
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    mla.selftest_wait_timeout(status, out)
    torch.cuda.synchronize()
    st, (waited_ms, ok) = int(status.item()), out.cpu().tolist()
    assert st & MLA_DEV_WAIT_TIMEOUT, st
    assert ok == 0
    assert 1900 <= waited_ms <= 10000, waited_ms  # the 2 s limit, give or take the polling step

    # the next calls run normally on the same context
    c = mi.decode_case(2, 1, 16, [128, 300], seed=0)
    o, lse, st2 = run_decode(c, 2)
    assert st2 == 0
    compare_decode(o, lse, *oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                                   c["seq_lens"], c["B"], c["Sq"], c["H"], c["scale"]))
