"""The failure path of the decode kernels, exercised without a fault.

GDN_FLAG_TEST_GIVE_UP makes the first wait for a state tile in every CTA give
up at once, as a wait that ran out of its time limit would. The kernel must
then wait (bounded) for the copies it still has in flight, write nothing more,
set bit 0 of the device error word and return. These tests check that the
call comes back well inside one wait's 2 s limit, that the error word reports
the give-up (and is cleared by reading it), and that the context stays usable:
the next ordinary call matches the oracle. Nothing faults, traps or hangs.
"""
import time

import numpy as np
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,L,T", [(4, 2, 1), (1, 1, 1), (4, 3, 4), (1, 1, 4), (4, 3, 12), (4, 3, 48)],
                         ids=["single_token", "single_token_small_launch", "one_chunk_window",
                              "window_small_launch", "multi_chunk_window", "tensor_core_window"])
def test_a_wait_that_gives_up_drains_reports_and_leaves_the_context_usable(cuda_device, B, L, T):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    h = W.host_inputs(w, threads=8)
    # an ordinary call first, so module loading is not part of the timed call
    warm = U.to_device(h, cuda_device)
    U.run_step(g, warm)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0

    t = U.to_device(h, cuda_device)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    U.run_step(g, t, flags=g.FLAG_TEST_GIVE_UP)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, f"the give-up path took {elapsed:.2f} s: a drain wait ran to its limit"
    assert g.gdn_read_device_error() == 1
    assert g.gdn_read_device_error() == 0  # reading clears the word

    fresh = U.to_device(h, cuda_device)
    y = U.run_step(g, fresh)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    ry, rs, rc = U.oracle_full(h)
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(fresh["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(fresh["conv_state"].cpu().numpy(), rc)
