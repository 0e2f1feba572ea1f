"""Calls captured in a CUDA graph and replayed give the same bits as direct
calls: the library allocates nothing, synchronises nothing and keeps no per-call
host state, so a decode step, and the mixer from the layer input (projections on
row-major or packed weights, then the step), can live inside a captured loop."""
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


# 3 x 2: the 3-CTA cluster kernel (one token and three); 4 x 2: the single-token kernel, the
# shared-memory window kernel
@pytest.mark.parametrize("B,T", [(3, 1), (4, 1), (3, 3), (4, 3)])
def test_graph_replay_equals_direct_calls(cuda_device, B, T):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=2, T=T)
    h = W.host_inputs(w, threads=8)
    direct = U.to_device(h, cuda_device)
    graphed = U.to_device(h, cuda_device)
    y_direct = torch.empty(direct["z"].shape, device=cuda_device)
    y_graph = torch.empty(graphed["z"].shape, device=cuda_device)

    def call(t, y):
        g.gdn_decode_step(t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
                          t["conv_state"], t["state"], y)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(graphed, y_graph)  # first call on the device does its one-time set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graphed["state"].copy_(torch.from_numpy(h["state"]))
    graphed["conv_state"].copy_(torch.from_numpy(h["conv_state"]))
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(graphed, y_graph)
    for _ in range(3):  # three decode steps: the state advances on every replay
        graph.replay()
        call(direct, y_direct)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y_direct)
    assert torch.equal(graphed["state"], direct["state"])
    assert torch.equal(graphed["conv_state"], direct["conv_state"])
    assert g.gdn_read_device_error() == 0


@pytest.mark.parametrize("packed", [False, True])
def test_graph_replay_of_the_mixer_equals_direct_calls(cuda_device, packed):
    """gdn_step_inputs (row-major or packed weights) then gdn_decode_step_ex with the gates
    ready, captured together in one graph: the replays give the bits of direct calls."""
    import numpy as np

    import gated_deltanet_linear_step_gb300 as g

    d = cuda_device
    E = 128
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=3, L=2, T=2)
    h = W.host_inputs(w, threads=8)
    ha = W.host_ab_inputs(w, E)
    wts = [W.proj_weights(w, l, E) for l in range(w.L)]

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(d).view(torch.bfloat16)

    wq = bf16(np.stack([x["w_qkv"] for x in wts]))
    wg = bf16(np.stack([x["w_gate"] for x in wts]))
    wa, wb = bf16(ha["w_alpha"]), bf16(ha["w_beta"])
    x = torch.from_numpy(ha["x"]).to(d)
    ws = torch.empty(g.gdn_in_proj_workspace_size(w.B, w.L, w.T, E), dtype=torch.uint8, device=d)
    pk = None
    if packed:
        pk = torch.empty(g.gdn_proj_pack_bytes(w.L, E), dtype=torch.uint8, device=d)
        g.gdn_pack_proj_weights(wq, wg, pk, wa, wb)

    def bufs():
        t = U.to_device(h, d)
        t["gate"] = torch.empty(t["alpha"].shape, device=d)
        t["betav"] = torch.empty(t["beta"].shape, device=d)
        t["y"] = torch.empty(t["z"].shape, device=d)
        return t

    def call(t):
        if pk is None:
            g.gdn_step_inputs(x, wq, wg, wa, wb, t["dt"], t["ssm_a"], t["qkv"], t["z"], t["gate"], t["betav"], ws)
        else:
            g.gdn_step_inputs_packed(x, pk, t["dt"], t["ssm_a"], t["qkv"], t["z"], t["gate"], t["betav"], ws)
        g.gdn_decode_step_ex(t["qkv"], t["z"], t["gate"], t["betav"], t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
                             t["conv_state"], t["state"], t["y"], flags=g.FLAG_GATES_READY)

    direct, graphed = bufs(), bufs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(graphed)  # one-time set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graphed["state"].copy_(torch.from_numpy(h["state"]))
    graphed["conv_state"].copy_(torch.from_numpy(h["conv_state"]))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(graphed)
    for _ in range(2):
        graph.replay()
        call(direct)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    for k in ("qkv", "z", "gate", "betav", "y", "state", "conv_state"):
        assert torch.equal(graphed[k], direct[k]), k
