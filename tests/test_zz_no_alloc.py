"""gdn_in_proj_noalloc: the input projections for callers that cannot allocate.

Some callers cannot hand the library a device workspace: a plug-in that only
receives tensors from a host framework whose allocator owns all device memory,
or code on a latency-critical path where a cudaMalloc would synchronise the
device. This entry point keeps the split of x in a fixed scratch array compiled
into the library instead. The size limit is a host-side check and is tested on
every machine; on a GPU the call is compared with the oracle and, on two calls
in a row with different sizes, bit for bit with gdn_in_proj on a caller
workspace (the second call finds the first call's contents in the shared array).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "gated_deltanet_linear_step_gb300", "libgdn.so")
SCRATCH = 48 << 20


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from gated_deltanet_linear_step_gb300 import _build

        _build.build()
    import gated_deltanet_linear_step_gb300 as g

    return g.load_library()


def _fake_pointers():
    base = 1 << 41  # aligned, non-overlapping values that are never dereferenced
    return [base, base + (1 << 32), base + (2 << 32), base + (3 << 32), base + (4 << 32)]


def test_noalloc_size_limit(lib):
    """Sizes beyond the scratch array are refused on the host, before any CUDA call."""
    p = _fake_pointers()
    # 256 x 36 x 1 tokens at n_embd 2560 need 94 MB of scratch: more than the library holds
    assert lib.gdn_in_proj_workspace_size(256, 36, 1, 2560) > SCRATCH
    assert lib.gdn_in_proj_noalloc(*p, 256, 36, 1, 2560, None) == 2
    assert b"scratch" in lib.gdn_last_error()
    assert lib.gdn_in_proj_noalloc(*p, 2, 3, 1, 100, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_noalloc_pointer_checks(lib):
    p = _fake_pointers()
    assert lib.gdn_in_proj_noalloc(p[0], None, *p[2:], 2, 3, 1, 128, None) == 1
    assert lib.gdn_in_proj_noalloc(*p[:4], p[3] + 16, 2, 3, 1, 128, None) == 4
    assert lib.gdn_in_proj_noalloc(p[0] + 4, *p[1:], 2, 3, 1, 128, None) == 3


def test_the_bench_and_verify_sizes_fit_the_scratch(lib):
    for B, L, T in ((64, 36, 1), (128, 36, 1), (16, 36, 8), (1, 36, 64)):
        assert 0 < lib.gdn_in_proj_workspace_size(B, L, T, 2560) <= SCRATCH


def _bf16(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def _inputs(B, L, T, E):
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    x = np.stack([np.stack([W.ab_x(w, b, l, E) for l in range(L)]) for b in range(B)])
    wts = [W.proj_weights(w, l, E) for l in range(L)]
    return x, np.stack([d["w_qkv"] for d in wts]), np.stack([d["w_gate"] for d in wts])


@pytest.mark.gpu
def test_noalloc_two_calls_in_a_row_match_the_workspace_call_and_the_oracle(cuda_device):
    import gated_deltanet_linear_step_gb300 as g

    E = 256
    # the second call has fewer token rows than the first, so it runs over the first call's scratch contents
    for B, L, T in ((3, 2, 5), (2, 2, 3)):
        x, wq, wg = _inputs(B, L, T, E)
        xd, wqd, wgd = torch.from_numpy(x).to(cuda_device), _bf16(wq, cuda_device), _bf16(wg, cuda_device)
        qkv = torch.full((B, L, T, W.CONV_CHANNELS), float("nan"), device=cuda_device)
        z = torch.full((B, L, T, W.VALUE_DIM), float("nan"), device=cuda_device)
        g.gdn_in_proj_noalloc(xd, wqd, wgd, qkv, z)
        qkv_ws, z_ws = torch.empty_like(qkv), torch.empty_like(z)
        ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
        g.gdn_in_proj(xd, wqd, wgd, qkv_ws, z_ws, ws)
        torch.cuda.synchronize()
        assert g.gdn_read_device_error() == 0
        assert torch.equal(qkv, qkv_ws) and torch.equal(z, z_ws)
        gq, gz = qkv.cpu().numpy().astype(np.float64), z.cpu().numpy().astype(np.float64)
        for l in range(L):
            rq, rz = oracle.in_proj(x[:, l], W.bf16_bits_to_float(wq[l]), W.bf16_bits_to_float(wg[l]))
            for gg, rr in ((gq[:, l], rq), (gz[:, l], rz)):
                gg = gg.reshape(-1, gg.shape[-1])
                rr = rr.reshape(-1, rr.shape[-1])
                assert np.max(np.abs(gg - rr).max(axis=1) / np.abs(rr).max(axis=1)) <= 1e-4


@pytest.mark.gpu
def test_noalloc_equals_the_workspace_call_at_the_bench_size(cuda_device):
    import gated_deltanet_linear_step_gb300 as g

    B, L, T, E = 64, 36, 1, 2560
    gen = torch.Generator(device=cuda_device).manual_seed(11)
    x = torch.randn((B, L, T, E), device=cuda_device, generator=gen)
    wq = (torch.randn((L, W.CONV_CHANNELS, E), device=cuda_device, generator=gen) * E ** -0.5).to(torch.bfloat16)
    wg = (torch.randn((L, W.VALUE_DIM, E), device=cuda_device, generator=gen) * E ** -0.5).to(torch.bfloat16)
    out = []
    for use_ws in (False, True):
        qkv = torch.empty((B, L, T, W.CONV_CHANNELS), device=cuda_device)
        z = torch.empty((B, L, T, W.VALUE_DIM), device=cuda_device)
        if use_ws:
            ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
            g.gdn_in_proj(x, wq, wg, qkv, z, ws)
        else:
            g.gdn_in_proj_noalloc(x, wq, wg, qkv, z)
        out.append((qkv, z))
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
