"""The step timeline build (libsdv_trace.so, sdv_trace_enable) on a tiny step:
every kernel of the step stamps its row, entry <= wait done <= exit, and each
kernel's wait for the kernel ahead ends after that kernel's exit (what
programmatic dependent launch guarantees)."""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

# prologue .. realignment, mma.sync paths at R = 6; stochastic verification
# from logits runs the draft tests inside the sampling kernel (no row 9)
STEP_ROWS = [0, 1, 2, 3, 4, 5, 6, 7, 8, 10, 11]


@pytest.fixture(scope="module")
def trace_engine():
    import torch
    assert torch.cuda.is_available()
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine, _abi, build
    from workloads import device as wd
    build.build(trace=True)
    W = wl.make_weights(wl.TINY, 1)
    eng = VerifyEngine(wd.config(wl.TINY, 3), wd.weights_to_device(W), 64, 8, lib_path=_abi.TRACE_LIB_PATH)
    return eng


def test_timeline_rows_and_order(trace_engine):
    import torch
    from workloads import device as wd
    eng = trace_engine
    batch = wl.workload1()
    table = torch.zeros((32, 3), dtype=torch.int64, device="cuda")
    table[:, 0:2] = 2 ** 62
    eng.set_trace(table)
    try:
        status, _, _ = gh.run_step(eng, batch, logits=False, probs=False)
    finally:
        eng.set_trace(None)
    assert status == 0
    t = table.cpu().numpy()
    prev_exit = None
    for k in STEP_ROWS:
        ent, wt, ex = (int(x) for x in t[k])
        assert 0 < ent <= wt <= ex, (k, ent, wt, ex)
        if prev_exit is not None:
            assert wt >= prev_exit, (k, wt, prev_exit)
        prev_exit = ex
    # points inside the sampling kernel, between its wait and its exit: every
    # block passes them in order and the slot's last block starts after every
    # block stored its chunk sums, so the first and the last arrival both rise
    smp_wait, smp_exit = int(t[10, 1]), int(t[10, 2])
    prev_first = prev_last = smp_wait
    for k in range(25, 31):
        first, last = int(t[k, 0]), int(t[k, 2])
        assert prev_first <= first <= last <= smp_exit and last >= prev_last, (k, first, last)
        prev_first, prev_last = first, last
    # rows of kernels the step does not launch stay as they were set
    assert t[9, 2] == 0 and (t[12:16, 2] == 0).all() and (t[16:25, 2] == 0).all() and (t[31:, 2] == 0).all()
    # stamps stop once the table is switched off
    before = table.clone()
    gh.run_step(eng, wl.workload1(), logits=False, probs=False)
    assert torch.equal(before, table)
