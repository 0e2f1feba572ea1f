"""GPU parity of the tensor-core input projections (qkv = w_qkv x, z = w_gate x)
against the oracle, and of the mixer step fed by them end to end."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu

# x is carried to within 2^-16 of its value (hi + lo halves), so the projection
# errors sit far below the 1e-4 bar; x rounded to BF16 alone would give ~1e-3.
SPLIT_TOL = 2e-5


def _bf16(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def _x(w, E):
    return np.stack([np.stack([W.ab_x(w, b, l, E) for l in range(w.L)]) for b in range(w.B)])


def _weights(w, E):
    wts = [W.proj_weights(w, l, E) for l in range(w.L)]
    return np.stack([d["w_qkv"] for d in wts]), np.stack([d["w_gate"] for d in wts])


def _guarded(shape, dev, guard=4096):
    """A NaN-filled buffer with `guard` floats on each side of the output view."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), float("nan"), device=dev)
    return buf, buf[guard:guard + n].view(*shape), guard


def _rows_rel_err(g, r):
    g = g.reshape(-1, g.shape[-1]).astype(np.float64)
    r = r.reshape(-1, r.shape[-1])
    return float(np.max(np.abs(g - r).max(axis=1) / np.abs(r).max(axis=1)))


def _oracle(x, wq, wg):
    B, L, T, _ = x.shape
    rq = np.empty((B, L, T, W.CONV_CHANNELS))
    rz = np.empty((B, L, T, W.VALUE_DIM))
    for l in range(L):
        rq[:, l], rz[:, l] = oracle.in_proj(x[:, l], W.bf16_bits_to_float(wq[l]), W.bf16_bits_to_float(wg[l]))
    return rq, rz


@pytest.mark.parametrize("B,L,T,E", [
    (3, 2, 5, 128),     # 15 tokens: one block of 16 rows, one padded row
    (1, 1, 1, 64),      # a single token and a single 64-wide slice
    (150, 1, 1, 64),    # two token blocks, the second ragged (22 of 128)
    (7, 2, 37, 256),    # 259 tokens: three blocks, the last 3 tokens
    (16, 1, 8, 2560),   # exactly 128 tokens, the model's n_embd
    (64, 2, 1, 2560),   # the batched-decode token count
])
def test_in_proj_matches_oracle(cuda_device, B, L, T, E):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    x = _x(w, E)
    wq, wg = _weights(w, E)
    qbuf, qkv, gq = _guarded((B, L, T, W.CONV_CHANNELS), cuda_device)
    zbuf, z, gz = _guarded((B, L, T, W.VALUE_DIM), cuda_device)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
    g.gdn_in_proj(torch.from_numpy(x).to(cuda_device), _bf16(wq, cuda_device), _bf16(wg, cuda_device), qkv, z, ws)
    assert g.gdn_read_device_error() == 0
    for buf, gd in ((qbuf, gq), (zbuf, gz)):
        assert torch.isnan(buf[:gd]).all() and torch.isnan(buf[-gd:]).all(), "write outside the output"
    gq_, gz_ = qkv.cpu().numpy(), z.cpu().numpy()
    assert not np.isnan(gq_).any() and not np.isnan(gz_).any(), "an output element was not written"
    rq, rz = _oracle(x, wq, wg)
    eq, ez = _rows_rel_err(gq_, rq), _rows_rel_err(gz_, rz)
    assert eq <= U.TOL and ez <= U.TOL, (eq, ez)
    assert max(eq, ez) <= SPLIT_TOL, (eq, ez)


def test_in_proj_is_deterministic(cuda_device):
    import gated_deltanet_linear_step_gb300 as g

    B, L, T, E = 5, 2, 3, 192
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    tx = torch.from_numpy(_x(w, E)).to(cuda_device)
    wq, wg = (_bf16(a, cuda_device) for a in _weights(w, E))
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
    outs = []
    for _ in range(2):
        qkv = torch.empty((B, L, T, W.CONV_CHANNELS), device=cuda_device)
        z = torch.empty((B, L, T, W.VALUE_DIM), device=cuda_device)
        g.gdn_in_proj(tx, wq, wg, qkv, z, ws)
        outs.append((qkv, z))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_in_proj_full_size_sampled(cuda_device):
    """The bench launch (64 sequences x 36 layers x 1 token, n_embd 2560). Layers 0, 17
    and 35 carry the seeded weights and are compared for sequences 0, 31 and 63; the
    other layers get other random weights and only load the kernel."""
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"]
    B, L, T, E = w.B, w.L, w.T, W.N_EMBD
    x = _x(w, E)
    gen = torch.Generator(device=cuda_device).manual_seed(7)
    wq = (torch.randn((L, W.CONV_CHANNELS, E), device=cuda_device, generator=gen) * E ** -0.5).to(torch.bfloat16)
    wg = (torch.randn((L, W.VALUE_DIM, E), device=cuda_device, generator=gen) * E ** -0.5).to(torch.bfloat16)
    layers, seqs = (0, 17, 35), (0, 31, 63)
    host = {}
    for l in layers:
        d = W.proj_weights(w, l, E)
        host[l] = d
        wq[l] = _bf16(d["w_qkv"], cuda_device)
        wg[l] = _bf16(d["w_gate"], cuda_device)
    qkv = torch.full((B, L, T, W.CONV_CHANNELS), float("nan"), device=cuda_device)
    z = torch.full((B, L, T, W.VALUE_DIM), float("nan"), device=cuda_device)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
    g.gdn_in_proj(torch.from_numpy(x).to(cuda_device), wq, wg, qkv, z, ws)
    assert g.gdn_read_device_error() == 0
    assert not torch.isnan(qkv).any().item() and not torch.isnan(z).any().item()
    for l in layers:
        rq, rz = oracle.in_proj(x[list(seqs), l], W.bf16_bits_to_float(host[l]["w_qkv"]),
                                W.bf16_bits_to_float(host[l]["w_gate"]))
        gq_ = qkv[list(seqs), l].cpu().numpy()
        gz_ = z[list(seqs), l].cpu().numpy()
        assert _rows_rel_err(gq_, rq) <= SPLIT_TOL and _rows_rel_err(gz_, rz) <= SPLIT_TOL


@pytest.mark.parametrize("B,L,T,E", [(3, 2, 5, 128), (150, 1, 1, 64), (16, 1, 8, 2560), (64, 2, 1, 2560)])
def test_step_inputs_match_oracle(cuda_device, B, L, T, E):
    """gdn_step_inputs: qkv and z as the oracle's in_proj, gate and beta as its ab_gates."""
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    x = _x(w, E)
    wq, wg = _weights(w, E)
    ha = W.host_ab_inputs(w, E)
    d = cuda_device
    outs = {}
    bufs = {}
    for name, width in (("qkv", W.CONV_CHANNELS), ("z", W.VALUE_DIM), ("gate", 48), ("beta", 48)):
        bufs[name], outs[name], gd = _guarded((B, L, T, width), d)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=d)
    g.gdn_step_inputs(torch.from_numpy(x).to(d), _bf16(wq, d), _bf16(wg, d), _bf16(ha["w_alpha"], d),
                      _bf16(ha["w_beta"], d), torch.from_numpy(ha["dt"]).to(d), torch.from_numpy(ha["ssm_a"]).to(d),
                      outs["qkv"], outs["z"], outs["gate"], outs["beta"], ws)
    assert g.gdn_read_device_error() == 0
    for name in outs:
        assert torch.isnan(bufs[name][:gd]).all() and torch.isnan(bufs[name][-gd:]).all(), name
        assert not torch.isnan(outs[name]).any().item(), name
    rq, rz = _oracle(x, wq, wg)
    assert _rows_rel_err(outs["qkv"].cpu().numpy(), rq) <= SPLIT_TOL
    assert _rows_rel_err(outs["z"].cpu().numpy(), rz) <= SPLIT_TOL
    rg = np.empty((B, L, T, 48))
    rb = np.empty((B, L, T, 48))
    for l in range(L):
        rg[:, l], rb[:, l] = oracle.ab_gates(x[:, l], ha["w_alpha_f32"][l], ha["w_beta_f32"][l], ha["dt"][l],
                                             ha["ssm_a"][l])
    assert _rows_rel_err(outs["gate"].cpu().numpy(), rg) <= U.TOL
    assert _rows_rel_err(outs["beta"].cpu().numpy(), rb) <= U.TOL


@pytest.mark.parametrize("T,fused", [(1, False), (3, False), (1, True), (3, True)])
def test_mixer_step_fed_by_the_projections(cuda_device, T, fused):
    """x -> gdn_in_proj + gdn_ab_gates (or gdn_step_inputs) -> gdn_decode_step_ex(GATES_READY)
    against the oracle's chain in_proj -> ab_gates -> gdn_decode. The conv history then
    holds projected values, which differ from the oracle's by the projection's rounding,
    so it is compared within the tolerance rather than bit for bit."""
    import gated_deltanet_linear_step_gb300 as g

    B, L, E = 2, 2, 256
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    h = W.host_inputs(w, threads=8)
    ha = W.host_ab_inputs(w, E)
    wq, wg = _weights(w, E)
    t = U.to_device(h, cuda_device)
    tx = torch.from_numpy(ha["x"]).to(cuda_device)
    qkv = torch.empty(t["qkv"].shape, device=cuda_device)
    z = torch.empty(t["z"].shape, device=cuda_device)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=cuda_device)
    gate = torch.empty(t["alpha"].shape, device=cuda_device)
    beta = torch.empty(t["beta"].shape, device=cuda_device)
    wa, wb = _bf16(ha["w_alpha"], cuda_device), _bf16(ha["w_beta"], cuda_device)
    if fused:
        g.gdn_step_inputs(tx, _bf16(wq, cuda_device), _bf16(wg, cuda_device), wa, wb, t["dt"], t["ssm_a"], qkv, z,
                          gate, beta, ws)
    else:
        g.gdn_in_proj(tx, _bf16(wq, cuda_device), _bf16(wg, cuda_device), qkv, z, ws)
        g.gdn_ab_gates(tx, wa, wb, t["dt"], t["ssm_a"], gate, beta)
    y = torch.empty(t["z"].shape, device=cuda_device)
    g.gdn_decode_step_ex(qkv, z, gate, beta, t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"], t["conv_state"],
                         t["state"], y, flags=g.FLAG_GATES_READY)
    assert g.gdn_read_device_error() == 0
    rq, rz = _oracle(ha["x"], wq, wg)
    rg = np.empty(h["alpha"].shape)
    rb = np.empty(h["beta"].shape)
    for l in range(L):
        rg[:, l], rb[:, l] = oracle.ab_gates(ha["x"][:, l], ha["w_alpha_f32"][l], ha["w_beta_f32"][l], h["dt"][l],
                                             h["ssm_a"][l])
    ry, rs, rc = oracle.gdn_decode(rq, rz, rg, rb, h["dt"], h["ssm_a"], h["conv_w"], h["ssm_norm"], h["conv_state"],
                                   h["state"], gates_ready=True)
    assert U.y_errors(y.cpu().numpy(), ry) <= U.TOL
    assert U.state_errors(t["state"].cpu().numpy(), rs) <= U.TOL
    gc = t["conv_state"].cpu().numpy().astype(np.float64)
    assert float(np.abs(gc - rc).max() / np.abs(rc).max()) <= U.TOL


def _packed_expected(wq, wg, wa, wb):
    """The packed layout restated in numpy: per layer 129 tiles of 128 rows (80 of w_qkv,
    48 of w_gate, then alpha, beta and 32 zero rows), per tile n_embd / 64 blocks of
    [128][64] BF16 where the 16-byte chunk c of row r sits at chunk position c XOR (r mod 8)."""
    L, _, E = wq.shape
    ab = np.zeros((L, 128, E), np.uint16)
    if wa is not None:
        ab[:, :48], ab[:, 48:96] = wa, wb
    rows = np.concatenate([wq, wg, ab], axis=1)              # [L][129 * 128][E]
    blocks = rows.reshape(L, 129, 128, E // 64, 8, 8)          # l, tile, r, ks, chunk, value
    blocks = blocks.transpose(0, 1, 3, 2, 4, 5).copy()         # l, tile, ks, r, chunk, value
    out = np.empty_like(blocks)
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    out[:, :, :, r, c ^ (r & 7)] = blocks[:, :, :, r, c]
    return out.reshape(-1).view(np.uint8)


@pytest.mark.parametrize("with_ab", [True, False])
def test_packed_weights_layout(cuda_device, with_ab):
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=1, L=2, T=1)
    E = 128
    wq, wg = _weights(w, E)
    ha = W.host_ab_inputs(w, E)
    d = cuda_device
    n = g.gdn_proj_pack_bytes(2, E)
    buf = torch.full((n + 2 * 4096,), 0xA5, dtype=torch.uint8, device=d)
    packed = buf[4096:4096 + n]
    wa = _bf16(ha["w_alpha"], d) if with_ab else None
    wb = _bf16(ha["w_beta"], d) if with_ab else None
    g.gdn_pack_proj_weights(_bf16(wq, d), _bf16(wg, d), packed, wa, wb)
    torch.cuda.synchronize()
    want = _packed_expected(wq.view(np.uint16), wg.view(np.uint16),
                            ha["w_alpha"].view(np.uint16) if with_ab else None,
                            ha["w_beta"].view(np.uint16) if with_ab else None)
    assert np.array_equal(packed.cpu().numpy(), want)
    assert (buf[:4096] == 0xA5).all() and (buf[-4096:] == 0xA5).all()


@pytest.mark.parametrize("B,L,T,E", [(3, 2, 5, 128), (150, 1, 1, 64), (64, 2, 1, 2560)])
def test_packed_projections_equal_unpacked_bit_for_bit(cuda_device, B, L, T, E):
    """gdn_in_proj_packed and gdn_step_inputs_packed feed the tensor cores the same values in
    the same order as the calls on the row-major weights: identical bits."""
    import gated_deltanet_linear_step_gb300 as g

    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=B, L=L, T=T)
    x = torch.from_numpy(_x(w, E)).to(cuda_device)
    wq, wg = _weights(w, E)
    ha = W.host_ab_inputs(w, E)
    d = cuda_device
    wq_d, wg_d = _bf16(wq, d), _bf16(wg, d)
    wa_d, wb_d = _bf16(ha["w_alpha"], d), _bf16(ha["w_beta"], d)
    dt, sa = torch.from_numpy(ha["dt"]).to(d), torch.from_numpy(ha["ssm_a"]).to(d)
    packed = torch.empty(g.gdn_proj_pack_bytes(L, E), dtype=torch.uint8, device=d)
    g.gdn_pack_proj_weights(wq_d, wg_d, packed, wa_d, wb_d)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=d)

    def outs():
        return {name: torch.full((B, L, T, width), float("nan"), device=d)
                for name, width in (("qkv", W.CONV_CHANNELS), ("z", W.VALUE_DIM), ("gate", 48), ("beta", 48))}

    a, b = outs(), outs()
    g.gdn_in_proj(x, wq_d, wg_d, a["qkv"], a["z"], ws)
    g.gdn_in_proj_packed(x, packed, b["qkv"], b["z"], ws)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    assert torch.equal(a["qkv"], b["qkv"]) and torch.equal(a["z"], b["z"])

    a, b = outs(), outs()
    g.gdn_step_inputs(x, wq_d, wg_d, wa_d, wb_d, dt, sa, a["qkv"], a["z"], a["gate"], a["beta"], ws)
    g.gdn_step_inputs_packed(x, packed, dt, sa, b["qkv"], b["z"], b["gate"], b["beta"], ws)
    torch.cuda.synchronize()
    assert g.gdn_read_device_error() == 0
    for name in a:
        assert not torch.isnan(b[name]).any().item(), name
        assert torch.equal(a[name], b[name]), name
