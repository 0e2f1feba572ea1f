"""HostDecodePipeline: steps fed from pinned host memory with overlapped copies give
the same bits as the same steps called directly on device tensors, step by step."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T", [("decode_b64_l36_t1", 1), ("verify_b16_l36_t8_ragged", 3)])
def test_pipeline_matches_direct_steps(cuda_device, name, T):
    import gated_deltanet_linear_step_gb300 as g
    from gated_deltanet_linear_step_gb300.host_pipeline import HostDecodePipeline

    w = W.WORKLOADS[name].scaled(B=3, L=2, T=T)
    h = W.host_inputs(w, threads=8)
    # five steps with different activations: each draws its own seeded inputs
    steps = [W.host_inputs(W.WORKLOADS[name].scaled(B=3, L=2, T=T, name=f"step{k}"), threads=8) for k in range(5)]
    for k, st in enumerate(steps):  # distinct per step: perturb deterministically
        for key in ("qkv", "z", "alpha", "beta"):
            st[key] = (st[key] * np.float32(1.0 + 0.1 * k)).astype(np.float32)

    # direct: device tensors, one call per step
    d = U.to_device(h, cuda_device)
    ys_direct = []
    for st in steps:
        for key in ("qkv", "z", "alpha", "beta"):
            d[key].copy_(torch.from_numpy(st[key]))
        y = torch.empty(d["z"].shape, device=cuda_device)
        if d["seq_len"] is None:
            g.gdn_decode_step(d["qkv"], d["z"], d["alpha"], d["beta"], d["dt"], d["ssm_a"], d["conv_w"],
                              d["ssm_norm"], d["conv_state"], d["state"], y)
        else:
            g.gdn_decode_step_varlen(d["qkv"], d["z"], d["alpha"], d["beta"], d["dt"], d["ssm_a"], d["conv_w"],
                                     d["ssm_norm"], d["conv_state"], d["state"], y, d["seq_len"])
        ys_direct.append(y.cpu())

    # pipelined: pinned host inputs, overlapped copies
    p = U.to_device(h, cuda_device)
    weights = {k: p[k] for k in ("dt", "ssm_a", "conv_w", "ssm_norm")}
    pipe = HostDecodePipeline(weights, p["conv_state"], p["state"], (w.B, w.L, w.T), seq_len=p["seq_len"])
    hosts = [{k: torch.from_numpy(st[k]).pin_memory() for k in ("qkv", "z", "alpha", "beta")} for st in steps]
    ys = [torch.empty(ys_direct[0].shape).pin_memory() for _ in steps]
    for k in range(len(steps)):
        pipe.submit(hosts[k], ys[k])
    pipe.synchronize()
    assert g.gdn_read_device_error() == 0
    # y of tokens past a sequence's length is not written by either path: compare valid tokens
    valid = torch.ones(ys_direct[0].shape[:3], dtype=torch.bool)
    if h["seq_len"] is not None:
        for b, n in enumerate(h["seq_len"]):
            valid[b, :, int(n):] = False
    for k in range(len(steps)):
        assert torch.equal(ys[k][valid], ys_direct[k][valid]), k
    assert torch.equal(p["state"], d["state"]) and torch.equal(p["conv_state"], d["conv_state"])
