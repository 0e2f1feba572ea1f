"""A decode call captured in a CUDA graph and replayed gives the same bits as
direct calls: the library allocates nothing, synchronises nothing and keeps no
per-call host state, so the call can live inside a captured decode loop."""
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 3])
def test_graph_replay_equals_direct_calls(cuda_device, T):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=3, L=2, T=T)
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
