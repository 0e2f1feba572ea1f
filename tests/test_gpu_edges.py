"""Edge cases of the decode step on the GPU: the longest window, lengths that are
negative, zero for every sequence, or zero in a single-token call, and activations
driven far into saturation."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _case(B, L, T, name="verify_b16_l36_t8_ragged"):
    w = W.WORKLOADS[name].scaled(B=B, L=L, T=T)
    return w, W.host_inputs(w, threads=8)


def test_longest_window_matches_oracle(cuda_device):
    """T at its maximum (1024 tokens, 16 chunks of the tensor-core kernel) against the oracle."""
    import gated_deltanet_linear_step_gb300 as g

    T = g.gdn_get_geometry()["max_t"]
    w, h = _case(1, 1, T, name="decode_b1_l36_t64_zero_state")
    t = U.to_device(h, cuda_device)
    y = U.run_step(g, t)
    assert g.gdn_read_device_error() == 0
    ry, rs, rc = U.oracle_full(h)
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)


# one token: 3 x 3 the single-token kernel, 3 x 1 the clusters; five tokens: 3 x 2 the clusters, 3 x 3 the
# shared-memory kernel
@pytest.mark.parametrize("L,T", [(3, 1), (1, 1), (2, 5), (3, 5), (2, 40)])
def test_negative_and_all_zero_lengths_change_nothing(cuda_device, L, T):
    import gated_deltanet_linear_step_gb300 as g

    w, h = _case(3, L, T)
    t = U.to_device(h, cuda_device)
    for lens in ([-7, 0, -1], [0, 0, 0]):
        t["seq_len"] = torch.tensor(lens, dtype=torch.int32, device=cuda_device)
        sentinel = torch.full(t["z"].shape, 777.0, device=cuda_device)
        y = U.run_step(g, t, y=sentinel.clone())
        torch.cuda.synchronize()
        assert g.gdn_read_device_error() == 0
        assert torch.equal(y, sentinel)
        assert torch.equal(t["state"].cpu(), torch.from_numpy(h["state"]))
        assert torch.equal(t["conv_state"].cpu(), torch.from_numpy(h["conv_state"]))


@pytest.mark.parametrize("B,L", [(4, 2), (3, 1)])
def test_single_token_call_with_lengths(cuda_device, B, L):
    """T = 1 runs the batched-decode kernel (4 x 2: 128 units) or, on a smaller launch (3 x 1: 48
    units, one round of clusters), the 3-CTA cluster kernel; a length of 0 leaves its sequence
    untouched and the others match the oracle."""
    import gated_deltanet_linear_step_gb300 as g

    w, h = _case(B, L, 1, name="decode_b64_l36_t1")
    h["seq_len"] = np.array([1, 0, 1, 0][:B], np.int32)
    t = U.to_device(h, cuda_device)
    sentinel = torch.full(t["z"].shape, -3.0, device=cuda_device)
    y = U.run_step(g, t, y=sentinel.clone())
    assert g.gdn_read_device_error() == 0
    ry, rs, rc = U.oracle_full(h)
    gy = y.cpu().numpy()
    for b in range(1, B, 2):
        assert np.all(gy[b] == -3.0)
        assert np.array_equal(t["state"][b].cpu().numpy(), h["state"][b])
    keep = list(range(0, B, 2))
    assert U.y_errors(gy[keep], ry[keep]) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)


@pytest.mark.parametrize("L,T,name", [(3, 1, "decode_b64_l36_t1"), (1, 1, "decode_b64_l36_t1"),
                                      (2, 5, "verify_b16_l36_t8_ragged"), (3, 5, "verify_b16_l36_t8_ragged"),
                                      (3, 20, "verify_b16_l36_t8_ragged"), (2, 40, "verify_b16_l36_t8_ragged")])
@pytest.mark.parametrize("gate", ["sigmoid", "silu"])
def test_saturated_activations_match_oracle(cuda_device, L, T, name, gate):
    """Inputs scaled so that SiLU, sigmoid and softplus see arguments far beyond +-88, where e^-x
    overflows or underflows in fp32: SiLU must go to x or 0, sigmoid to 1 or 0, beta to 0 or 1 and
    decay to 0 or 1, as in the fp64 oracle. Covers the single-token kernel (3 x 3 x 1), the 3-CTA
    cluster kernel (3 x 1 x 1, 3 x 2 x 5), the shared-memory kernel (3 x 3 x 5 and 20) and the
    tensor-core kernel."""
    import gated_deltanet_linear_step_gb300 as g

    w, h = _case(3, L, T, name=name)
    for k, f in (("qkv", 120.0), ("conv_state", 120.0), ("z", 150.0), ("alpha", 60.0), ("beta", 60.0)):
        h[k] = (h[k] * np.float32(f)).astype(np.float32)
    t = U.to_device(h, cuda_device)
    flags = g.FLAG_SILU_GATE if gate == "silu" else 0
    y = U.run_step(g, t, flags=flags)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    with np.errstate(over="ignore"):
        ry, rs, rc = U.oracle_full(h, gate=gate)
    gy = y.cpu().numpy()
    assert np.all(np.isfinite(gy[~np.isnan(ry)]))
    assert U.y_errors(gy, ry) <= U.TOL
    # With beta and decay both driven to zero the fp64 oracle keeps tiles near 1e-50, which fp32
    # cannot hold: 1e-4 relative needs 14 significant bits, which fp32 has only above about 2^-112.
    # Tiles whose oracle magnitude is below 2^-100 must come out below 2^-100; the rest meet the bar.
    gs = t["state"].cpu().numpy().reshape(-1, 128 * 128).astype(np.float64)
    rt = rs.reshape(-1, 128 * 128)
    floor = 2.0 ** -100
    tiny = np.abs(rt).max(axis=1) < floor
    assert np.all(np.abs(gs[tiny]).max(axis=1) < floor)
    assert U.state_errors(gs[~tiny], rt[~tiny]) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)
