"""GPU parity of the fused alpha/beta projection with its gate epilogue, and of
the decode step fed with its outputs (GDN_FLAG_GATES_READY), against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _device_ab(h, dev):
    t = {k: torch.from_numpy(np.ascontiguousarray(h[k])).to(dev) for k in ("x", "dt", "ssm_a")}
    for k in ("w_alpha", "w_beta"):
        t[k] = torch.from_numpy(h[k].view(np.int16)).to(dev).view(torch.bfloat16)
    return t


def _rows_rel_err(g, r):
    g = g.reshape(-1, g.shape[-1]).astype(np.float64)
    r = r.reshape(-1, r.shape[-1])
    return float(np.max(np.abs(g - r).max(axis=1) / np.abs(r).max(axis=1)))


# n_embd 768 and 1280 give each rank of the cluster 3 and 5 64-wide units: a 128-wide slice
# followed by a 64-wide tail in one double buffer; 33 rows also end in a partial second row block.
@pytest.mark.parametrize("B,L,T,E", [(3, 2, 1, 2560), (2, 3, 5, 2560), (17, 1, 1, 128), (1, 1, 33, 64), (64, 2, 1, 2560),
                                     (5, 2, 3, 768), (33, 1, 1, 1280)])
def test_ab_gates_match_oracle(cuda_device, B, L, T, E):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    h = W.host_ab_inputs(w, E)
    t = _device_ab(h, cuda_device)
    gate = torch.full((B, L, T, 48), float("nan"), device=cuda_device)
    beta = torch.full((B, L, T, 48), float("nan"), device=cuda_device)
    g.gdn_ab_gates(t["x"], t["w_alpha"], t["w_beta"], t["dt"], t["ssm_a"], gate, beta)
    torch.cuda.synchronize()
    rg = np.empty((B, L, T, 48))
    rb = np.empty((B, L, T, 48))
    for l in range(L):
        rg[:, l], rb[:, l] = oracle.ab_gates(h["x"][:, l], h["w_alpha_f32"][l], h["w_beta_f32"][l], h["dt"][l],
                                             h["ssm_a"][l])
    assert _rows_rel_err(gate.cpu().numpy(), rg) <= U.TOL
    assert _rows_rel_err(beta.cpu().numpy(), rb) <= U.TOL


# 2 x 2: the 3-CTA cluster kernel for one token and four; 4 x 2: the single-token kernel and the
# shared-memory window kernel; 36 tokens: the tensor-core kernel
@pytest.mark.parametrize("B,T", [(2, 1), (4, 1), (2, 4), (4, 4), (2, 36)])
def test_step_fed_by_ab_gates_matches_oracle(cuda_device, B, T):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=2, T=T)
    h = W.host_inputs(w, threads=8)
    ha = W.host_ab_inputs(w)
    t = U.to_device(h, cuda_device)
    ta = _device_ab(ha, cuda_device)
    gate = torch.empty(t["alpha"].shape, device=cuda_device)
    beta = torch.empty(t["beta"].shape, device=cuda_device)
    g.gdn_ab_gates(ta["x"], ta["w_alpha"], ta["w_beta"], t["dt"], t["ssm_a"], gate, beta)
    y = torch.empty(t["z"].shape, device=cuda_device)
    g.gdn_decode_step_ex(t["qkv"], t["z"], gate, beta, t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
                         t["conv_state"], t["state"], y, flags=g.FLAG_GATES_READY)
    torch.cuda.synchronize()
    rg = np.empty(h["alpha"].shape)
    rb = np.empty(h["beta"].shape)
    for l in range(w.L):
        rg[:, l], rb[:, l] = oracle.ab_gates(ha["x"][:, l], ha["w_alpha_f32"][l], ha["w_beta_f32"][l], h["dt"][l],
                                             h["ssm_a"][l])
    ry, rs, rc = oracle.gdn_decode(h["qkv"], h["z"], rg, rb, h["dt"], h["ssm_a"], h["conv_w"], h["ssm_norm"],
                                   h["conv_state"], h["state"], gates_ready=True)
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)
