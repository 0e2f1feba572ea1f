"""The recurrent state around the kernel: the conv-history hazard between the v
heads of a k head, and checkpoint/resume of state and conv_state."""
import io

import numpy as np
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,L,T", [(4, 2, 1), (1, 2, 1), (2, 2, 3), (4, 2, 3), (2, 2, 20), (4, 2, 20), (2, 2, 40),
                                   (2, 2, 70)])
def test_every_v_head_of_a_k_head_sees_the_old_conv_history(cuda_device, B, L, T):
    """The q/k conv history of head g is read by the work of all three v heads 3g..3g+2 and
    rolled once. Old history entries 1000x larger than any new input make a read of the
    rolled history by any of the three show up as a y error far above the tolerance. (4 x 2 runs
    the single-token kernel for one token and the shared-memory kernel for windows; 1 x 2 x 1 and
    2 x 2 x 3 the 3-CTA cluster kernel, where the three v heads are on three CTAs.)"""
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    h = W.host_inputs(w, threads=8)
    qk_channels = 2 * W.K_HEADS * W.HEAD_DIM  # q and k: channels [0, 4096)
    h["conv_state"][:, :, :qk_channels, :] *= np.float32(1000.0)
    t = U.to_device(h, cuda_device)
    y = U.run_step(g, t)
    assert g.gdn_read_device_error() == 0
    with np.errstate(over="ignore"):  # SiLU of conv outputs near -1e4: exp overflows to inf, the limit is exact
        ry, rs, rc = U.oracle_full(h)
    gy = y.cpu().numpy()
    for vh in range(48):  # every v head on its own, all three of each k head
        sl = slice(vh * 128, (vh + 1) * 128)
        err = np.abs(gy[..., sl] - ry[..., sl]).max() / np.abs(ry[..., sl]).max()
        assert err <= U.TOL, (vh, err)
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)


@pytest.mark.parametrize("T", [1, 4])
def test_checkpoint_and_resume_equal_an_uninterrupted_run(cuda_device, T):
    """Three calls in a row against two calls, a save of state and conv_state through
    torch.save, a reload into fresh tensors, and the third call: identical bits."""
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=2, L=2, T=T)
    h = W.host_inputs(w, threads=8)
    a = U.to_device(h, cuda_device)
    ys = [U.run_step(g, a) for _ in range(3)]
    b = U.to_device(h, cuda_device)
    for _ in range(2):
        U.run_step(g, b)
    buf = io.BytesIO()
    torch.save({"state": b["state"].cpu(), "conv_state": b["conv_state"].cpu()}, buf)
    buf.seek(0)
    ck = torch.load(buf)
    c = U.to_device(h, cuda_device)
    c["state"].copy_(ck["state"])
    c["conv_state"].copy_(ck["conv_state"])
    y3 = U.run_step(g, c)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    assert torch.equal(y3, ys[2])
    assert torch.equal(c["state"], a["state"]) and torch.equal(c["conv_state"], a["conv_state"])
