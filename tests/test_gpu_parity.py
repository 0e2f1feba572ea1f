"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases are compared element by element on every output; they span
several tiles, several 8-token chunks and ragged tails. The five workloads at
full size run in the launch configuration ``bench.py`` times and are compared
on sampled (sequence, layer) slices, which the oracle regenerates from the
seed on its own; conv_state is checked bit-exactly on every slice. Tolerances
are in ``tests/parity_util.py``: 1e-4 normwise relative on y and on the state.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(cuda_device):
    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    yield g
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0


SMALL = [
    ("decode_b1_l1_t1", {}),                         # one token, 16 units: the 3-CTA cluster kernel
    ("decode_b64_l36_t1", dict(B=1, L=3)),           # one token, 48 units: that kernel
    ("decode_b64_l36_t1", dict(B=3, L=2)),           # one token, 96 units: that kernel
    ("decode_b64_l36_t1", dict(B=4, L=2)),           # one token, 128 units: the single-token kernel
    ("decode_b64_l36_t1", dict(B=10, L=1)),          # one token, 160 units: the clusters again, two rounds
    ("decode_b128_l36_t1_beta_hi_decay_hi", dict(B=2, L=2)),
    ("verify_b16_l36_t8_ragged", dict(B=6, L=2)),   # windows of 2-23 tokens over more than 97 units: the
    ("decode_b1_l36_t64_zero_state", dict(L=2)),    # shared-memory kernel in 8-token chunks; up to 97, the
    ("decode_b64_l36_t1", dict(B=2, L=1, T=2)),     # 3-CTA cluster kernel (one round of clusters)
    ("decode_b64_l36_t1", dict(B=2, L=4, T=2)),
    ("decode_b64_l36_t1", dict(B=2, L=1, T=3)),
    ("decode_b64_l36_t1", dict(B=2, L=4, T=3)),
    ("decode_b64_l36_t1", dict(B=1, L=2, T=9)),
    ("decode_b64_l36_t1", dict(B=1, L=8, T=9)),
    ("decode_b64_l36_t1", dict(B=2, L=1, T=17)),
    ("decode_b64_l36_t1", dict(B=2, L=4, T=17)),
    ("verify_b16_l36_t8_ragged", dict(B=5, L=1, T=20)),
    ("verify_b16_l36_t8_ragged", dict(B=5, L=2, T=20)),
    ("decode_b64_l36_t1", dict(B=2, L=1, T=23)),
    ("decode_b64_l36_t1", dict(B=2, L=4, T=23)),   # two full 8-token chunks and 7 tokens, the longest on that kernel
    ("decode_b64_l36_t1", dict(B=2, L=1, T=24)),   # the shortest window on the tensor-core kernel
    ("decode_b64_l36_t1", dict(B=2, L=1, T=25)),
    ("decode_b64_l36_t1", dict(B=2, L=1, T=40)),
    ("decode_b128_l36_t1_beta_hi_decay_hi", dict(B=1, L=1, T=64)),
    ("verify_b16_l36_t8_ragged", dict(B=5, L=1, T=70)),
]


@pytest.mark.parametrize("name,scale", SMALL, ids=[f"{n}-{s}" for n, s in SMALL])
def test_small_cases_match_oracle_elementwise(g, name, scale):
    w = W.WORKLOADS[name].scaled(**scale)
    h = W.host_inputs(w, threads=8)
    t = U.to_device(h, torch.device("cuda:0"))
    y = U.run_step(g, t)
    torch.cuda.synchronize()
    ry, rs, rc = U.oracle_full(h)
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)


@pytest.mark.parametrize("L", [2, 3])  # 96 units: the 3-CTA clusters; 144: the shared-memory kernel
def test_silu_gate_variant_matches_oracle(g, L):
    w = W.WORKLOADS["verify_b16_l36_t8_ragged"].scaled(B=3, L=L)
    h = W.host_inputs(w, threads=8)
    t = U.to_device(h, torch.device("cuda:0"))
    y = U.run_step(g, t, flags=g.FLAG_SILU_GATE)
    torch.cuda.synchronize()
    ry, rs, rc = U.oracle_full(h, gate="silu")
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(t["conv_state"].cpu().numpy(), rc)


FULL = {
    "decode_b1_l1_t1": [(0, 0)],
    "decode_b1_l36_t64_zero_state": [(0, 0), (0, 17), (0, 35)],
    "decode_b64_l36_t1": [(0, 0), (63, 35), (31, 17), (5, 30), (40, 1), (17, 22)],
    "decode_b128_l36_t1_beta_hi_decay_hi": [(0, 0), (127, 35), (64, 18), (3, 33), (99, 7)],
    "verify_b16_l36_t8_ragged": "by_length",
}


def test_multi_chunk_window_at_full_layer_count(g):
    """A 16-token window (two 8-token chunks on the shared-memory kernel) over 16 sequences and all
    36 layers, in the launch configuration of the benchmarked windows, on sampled slices."""
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=16, T=16)
    dev = torch.device("cuda:0")
    t = W.device_inputs(w, dev, threads=16)
    y = torch.full(t["z"].shape, float("nan"), device=dev)
    U.run_step(g, t, y=y)
    torch.cuda.synchronize()
    for b, l in [(0, 0), (15, 35), (7, 18), (11, 3)]:
        ry, rs, rc = U.oracle_slice(w, b, l)
        gy, gs = y[b, l].cpu().numpy(), t["state"][b, l].cpu().numpy()
        assert U.y_errors(gy, ry) <= U.TOL, (b, l)
        assert U.state_errors(gs, rs) <= U.TOL, (b, l)
        assert np.array_equal(t["conv_state"][b, l].cpu().numpy(), rc), (b, l)
    assert torch.isfinite(t["state"]).all()


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workloads_on_sampled_slices(g, name):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda:0")
    t = W.device_inputs(w, dev, threads=16)
    cs_before = t["conv_state"].cpu().numpy()
    qkv = t["qkv"].cpu().numpy()
    y = torch.full(t["z"].shape, float("nan"), device=dev)
    U.run_step(g, t, y=y)
    torch.cuda.synchronize()
    lens = W.seq_lens(w)
    samples = FULL[name]
    if samples == "by_length":
        # one sequence per distinct length, at two layers each
        firsts = {int(n): b for b, n in reversed(list(enumerate(lens)))}
        samples = [(b, l) for b in sorted(firsts.values()) for l in (0, 29)]
    for b, l in samples:
        ry, rs, rc = U.oracle_slice(w, b, l)
        gy, gs = y[b, l].cpu().numpy(), t["state"][b, l].cpu().numpy()
        print(U.report(f"{name} b={b} l={l}", gy, ry, gs, rs))
        assert U.y_errors(gy, ry) <= U.TOL, (b, l)
        assert U.state_errors(gs, rs) <= U.TOL, (b, l)
        assert np.array_equal(t["conv_state"][b, l].cpu().numpy(), rc), (b, l)
    # every slice: conv_state is the last three inputs of [old history, valid tokens]
    cs = t["conv_state"].cpu().numpy()
    for b in range(w.B):
        n = w.T if lens is None else int(lens[b])
        hist = np.concatenate([cs_before[b], np.moveaxis(qkv[b, :, :n], 1, 2)], axis=2)
        assert np.array_equal(cs[b], hist[..., -3:]), b
    assert torch.isfinite(t["state"]).all()


def _small(scale=dict(B=3, L=2, T=9), name="verify_b16_l36_t8_ragged"):
    w = W.WORKLOADS[name].scaled(**scale)
    return w, W.host_inputs(w, threads=8)


@pytest.mark.parametrize("L", [2, 3])
def test_t_tokens_in_one_call_equal_t_single_calls(g, L):
    """One T-token call and T one-token calls agree to within the parity tolerance:
    both follow the same definition, but the window kernels regroup it by chunks (in
    fp32 up to 23 tokens; past that with the products on the tensor cores, BF16 hi + lo
    operands, errors near 2e-5 of the largest value), while the single-token kernel
    sums token by token."""
    w, h = _small(dict(B=3, L=L, T=9), name="decode_b64_l36_t1")
    dev = torch.device("cuda:0")
    a = U.to_device(h, dev)
    ya = U.run_step(g, a)
    b = U.to_device(h, dev)
    ys = []
    for tt in range(w.T):
        one = dict(b)
        for k in ("qkv", "z", "alpha", "beta"):
            one[k] = b[k][:, :, tt:tt + 1].contiguous()
        ys.append(U.run_step(g, one))
    torch.cuda.synchronize()
    assert U.y_errors(ya.cpu().numpy(), torch.cat(ys, dim=2).cpu().numpy().astype("float64")) <= U.TOL
    assert U.state_errors(a["state"].cpu().numpy(), b["state"].cpu().numpy().astype("float64")) <= U.TOL
    assert torch.equal(a["conv_state"], b["conv_state"])


# (window length, prefix length, layers): both calls of a case run the same kernel over the same
# chunks, so they agree bit for bit: up to 23 tokens the 3-CTA cluster kernel at 2 layers (the
# prefix call's single sequence too), the shared-memory kernel in chunks of 8 at 7 layers (112 units
# for the single sequence); 25 or more the tensor-core kernel in chunks of 64.
@pytest.mark.parametrize("T,P,L", [(8, 3, 2), (8, 3, 7), (12, 10, 2), (12, 10, 7), (40, 33, 2), (70, 66, 2)])
def test_ragged_equals_prefix_and_leaves_invalid_steps_untouched(g, T, P, L):
    w, h = _small(dict(B=3, L=L, T=T))
    dev = torch.device("cuda:0")
    lens = torch.tensor([0, P, T], dtype=torch.int32, device=dev)
    a = U.to_device(h, dev)
    a["seq_len"] = lens
    sentinel = torch.full(a["z"].shape, 12345.0, device=dev)
    ya = U.run_step(g, a, y=sentinel.clone())
    torch.cuda.synchronize()
    # sequence 0: nothing written
    assert torch.equal(ya[0], sentinel[0])
    assert torch.equal(a["state"][0], torch.from_numpy(h["state"][0]).to(dev))
    assert torch.equal(a["conv_state"][0], torch.from_numpy(h["conv_state"][0]).to(dev))
    # sequence 1: the prefix call with T = P
    p = U.to_device(h, dev)
    p = {k: (v[1:2] if v is not None and k not in ("dt", "ssm_a", "conv_w", "ssm_norm") else v) for k, v in p.items()}
    for k in ("qkv", "z", "alpha", "beta"):
        p[k] = p[k][:, :, :P].contiguous()
    p["seq_len"] = None
    yp = U.run_step(g, p)
    torch.cuda.synchronize()
    assert torch.equal(ya[1, :, :P], yp[0]) and torch.equal(ya[1, :, P:], sentinel[1, :, P:])
    assert torch.equal(a["state"][1], p["state"][0]) and torch.equal(a["conv_state"][1], p["conv_state"][0])
    # lengths past T are clamped to T
    c = U.to_device(h, dev)
    c["seq_len"] = torch.tensor([100, T, T], dtype=torch.int32, device=dev)
    yc = U.run_step(g, c)
    full = U.to_device(h, dev)
    yf = U.run_step(g, full, seq_len=None)
    torch.cuda.synchronize()
    assert torch.equal(yc, yf) and torch.equal(c["state"], full["state"])
    assert torch.equal(yc[2], ya[2]) and torch.equal(c["state"][2], a["state"][2])
    # and the ragged call matches the oracle
    ry, rs, _ = U.oracle_full(dict(h, seq_len=lens.cpu().numpy()))
    assert U.y_errors(np.where(np.isnan(ry), np.nan, ya.cpu().numpy()), ry) <= U.TOL
    assert U.state_errors(a["state"].cpu().numpy(), rs) <= U.TOL


@pytest.mark.parametrize("L", [2, 1])  # 128 units: the shared-memory kernel; 64: the 3-CTA clusters
def test_deterministic_and_batch_permutation_equivariant(g, L):
    w, h = _small(dict(B=4, L=L, T=3), name="decode_b64_l36_t1")
    dev = torch.device("cuda:0")
    a = U.to_device(h, dev)
    ya = U.run_step(g, a)
    b = U.to_device(h, dev)
    yb = U.run_step(g, b)
    perm = [2, 0, 3, 1]
    hp = {k: (v[perm] if v is not None and v.shape[0] == 4 and k not in ("dt", "ssm_a", "conv_w", "ssm_norm")
              else v) for k, v in h.items()}
    c = U.to_device(hp, dev)
    yc = U.run_step(g, c)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a["state"], b["state"])
    assert torch.equal(yc, ya[perm]) and torch.equal(c["state"], a["state"][perm])
    assert torch.equal(c["conv_state"], a["conv_state"][perm])


@pytest.mark.parametrize("T,L", [(6, 2), (6, 3), (16, 2), (16, 3), (40, 2)])
def test_verify_window_then_commit(g, T, L):
    w, h = _small(dict(B=3, L=L, T=T))
    dev = torch.device("cuda:0")
    win = U.to_device(h, dev)
    y = torch.full(win["z"].shape, float("nan"), device=dev)
    g.gdn_verify_window(win["qkv"], win["z"], win["alpha"], win["beta"], win["dt"], win["ssm_a"], win["conv_w"],
                        win["ssm_norm"], win["conv_state"], win["state"], y)
    ref = U.to_device(h, dev)
    yref = U.run_step(g, ref, seq_len=None)
    torch.cuda.synchronize()
    # phase 1: the same y as a full decode, with both states untouched
    assert torch.equal(y, yref)
    assert torch.equal(win["state"], torch.from_numpy(h["state"]).to(dev))
    assert torch.equal(win["conv_state"], torch.from_numpy(h["conv_state"]).to(dev))
    # phase 2: keep 2, T and 0 tokens
    n_keep = torch.tensor([2, T, 0], dtype=torch.int32, device=dev)
    g.gdn_verify_commit(win["qkv"], win["alpha"], win["beta"], win["dt"], win["ssm_a"], win["conv_w"],
                        win["conv_state"], win["state"], n_keep)
    exp = U.to_device(h, dev)
    U.run_step(g, exp, seq_len=n_keep)
    torch.cuda.synchronize()
    assert torch.equal(win["state"], exp["state"]) and torch.equal(win["conv_state"], exp["conv_state"])
    _, rs, rc = U.oracle_full(dict(h, seq_len=n_keep.cpu().numpy()))
    assert U.state_errors(win["state"].cpu().numpy(), rs) <= U.TOL
    assert np.array_equal(win["conv_state"].cpu().numpy(), rc)


@pytest.mark.parametrize("B,L", [(1, 1), (4, 2)])  # the 3-CTA clusters, the shared-memory kernel
def test_outputs_have_untouched_guard_regions(g, B, L):
    w, h = _small(dict(B=B, L=L, T=3), name="decode_b64_l36_t1")
    dev = torch.device("cuda:0")
    t = U.to_device(h, dev)
    pad = 64  # floats = 256 bytes on each side
    bufs = {}
    for k in ("state", "conv_state"):
        n = t[k].numel()
        big = torch.full((n + 2 * pad,), float("nan"), device=dev)
        big[pad:pad + n] = t[k].reshape(-1)
        bufs[k] = big
        t[k] = big[pad:pad + n].view(t[k].shape)
    ny = t["z"].numel()
    ybig = torch.full((ny + 2 * pad,), float("nan"), device=dev)
    y = ybig[pad:pad + ny].view(t["z"].shape)
    U.run_step(g, t, y=y)
    torch.cuda.synchronize()
    for big in list(bufs.values()) + [ybig]:
        assert torch.isnan(big[:pad]).all() and torch.isnan(big[-pad:]).all()
    assert torch.isfinite(y).all()


def test_bad_arguments_raise_and_launch_nothing(g):
    w, h = _small(dict(B=1, L=1, T=2), name="decode_b64_l36_t1")
    dev = torch.device("cuda:0")
    t = U.to_device(h, dev)
    before = t["state"].clone()
    y = torch.zeros(t["z"].shape, device=dev)
    args = [t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
            t["conv_state"], t["state"], y]
    lib = g.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    ptrs = [a.data_ptr() for a in args]
    # misaligned state pointer, y aliasing state, y aliasing qkv, null conv_state
    for i, val, code in [(9, ptrs[9] + 4, 3), (10, ptrs[9], 4), (10, ptrs[0], 4), (8, None, 1)]:
        p = list(ptrs)
        p[i] = val
        assert lib.gdn_decode_step(*p, 1, 1, 2, stream) == code
    with pytest.raises(g.GdnError):
        g.gdn_decode_step_ex(*args, flags=0x100)
    with pytest.raises(ValueError):
        g.gdn_decode_step(*args[:10], torch.zeros(1, 1, 3, 6144, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(t["state"], before) and torch.all(y == 0)


@pytest.mark.parametrize("B,L,T", [(4, 2, 1), (1, 2, 1), (3, 2, 4), (4, 2, 4), (3, 2, 12), (4, 2, 12), (3, 2, 40),
                                   (3, 2, 70)])
def test_no_y_and_no_state_write_flags_match_the_full_call(g, B, L, T):
    """FLAG_NO_Y gives the full call's state and conv_state bit for bit and writes no y;
    FLAG_NO_STATE_WRITE gives its y bit for bit and leaves both states untouched. (One token: 4 x 2
    runs the single-token kernel, 1 x 2 the 3-CTA cluster kernel; windows up to 23 tokens: 3 x 2 the
    cluster kernel, 4 x 2 the shared-memory kernel.)"""
    w, h = _small(dict(B=B, L=L, T=T), name="decode_b64_l36_t1")
    dev = torch.device("cuda:0")
    full = U.to_device(h, dev)
    yf = U.run_step(g, full, seq_len=None)
    a = U.to_device(h, dev)
    sentinel = torch.full(a["z"].shape, 777.0, device=dev)
    ya = U.run_step(g, a, y=sentinel.clone(), seq_len=None, flags=g.FLAG_NO_Y)
    b = U.to_device(h, dev)
    yb = U.run_step(g, b, seq_len=None, flags=g.FLAG_NO_STATE_WRITE)
    torch.cuda.synchronize()
    assert torch.equal(ya, sentinel)
    assert torch.equal(a["state"], full["state"]) and torch.equal(a["conv_state"], full["conv_state"])
    assert torch.equal(yb, yf)
    assert torch.equal(b["state"], torch.from_numpy(h["state"]).to(dev))
    assert torch.equal(b["conv_state"], torch.from_numpy(h["conv_state"]).to(dev))


def test_dispatch_query_names_the_kernel_of_each_size(g):
    """gdn_dispatch_kernel gives the kernel the library runs; on unambiguous sizes it agrees with the
    rules as bench.py states them (which the bench uses only without a GPU)."""
    import bench

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = {(1, 1, 1): "gdn_window_kernel", (4, 1, 1): "gdn_window_kernel", (4, 2, 1): "gdn_decode_t1_kernel",
             (64, 36, 1): "gdn_decode_t1_kernel", (2, 1, 8): "gdn_window_kernel", (16, 36, 8): "gdn_chunk_kernel",
             (1, 36, 64): "gdn_window_tc_kernel", (2, 1, 24): "gdn_window_tc_kernel", (4, 2, 23): "gdn_chunk_kernel"}
    for (B, L, T), want in cases.items():
        got = g.gdn_dispatch_kernel(B, L, T)
        assert got == want, (B, L, T, got)
        assert got == bench.kernel_name(T, B * L * 16, sms), (B, L, T)
    with pytest.raises(g.GdnError):
        g.gdn_dispatch_kernel(0, 1, 1)
