"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up after its limit, the kernel returns, gdn_check_status reports
GDN_ETIMEOUT once, and the context stays usable (a forward afterwards passes
parity)."""
import time

import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
from chunkwise_gated_deltanet_gb300 import gdn as binding
import workloads
from tests.parity import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_unsatisfied_wait_reports_timeout_and_context_survives():
    gdn.gdn_check_status()  # start from a clear status word
    t0 = time.perf_counter()
    binding.gdn_selftest_wait_timeout()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_check_status()
    waited = time.perf_counter() - t0
    assert e.value.status == binding.GDN_ETIMEOUT
    assert 1.5 < waited < 30.0, waited  # the kernels' wait limit is 2 s
    gdn.gdn_check_status()  # the word was cleared by the read
    inp = workloads.make_inputs(workloads.WORKLOADS["gdn_bf16_b4h16t4096d128c64"], B=1, H=2,
                                T=130)
    o, s = run_gpu(inp, 64)
    ro, rs = run_oracle(inp)
    assert_close(o, ro, False, "out after the timeout", stored_bf16=True)
    assert_close(s, rs, False, "S_final after the timeout")
