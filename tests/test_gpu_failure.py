"""Device-side failure detection without a GPU fault: the bounded mbarrier wait
used by the TMA-fed and tensor-core kernels gives up on a barrier that nothing
completes, records ZETA_ERR_DEVICE_TIMEOUT in the status word, and the context
stays usable for the next calls."""
import numpy as np
import pytest
import torch

from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W

from gpu_util import Run

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def test_wait_that_runs_out_reports_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zb.zeta_check_bounded_wait(2000, 0, st)              # nothing completes the barrier
    torch.cuda.synchronize()
    assert int(st.item()) == 5                            # ZETA_ERR_DEVICE_TIMEOUT


def test_completed_barrier_is_not_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zb.zeta_check_bounded_wait(2000, 1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_context_usable_after_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zb.zeta_check_bounded_wait(100, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5
    run = Run(W.TINY.replace(N=256, C=64, k=8))
    assert run.status() == 0
    assert np.isfinite(run.out()).all()
