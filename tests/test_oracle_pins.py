"""Pins of the fp64 oracle to facts other than itself.

Each test checks the oracle against something the pages or the mathematics
fix independently: the page's constants (``tests/golden/geometry.txt``),
closed forms, exact rational arithmetic on tiny inputs, element-by-element
recomputation with ``math`` routines, and invariants of the definition
(operation order from the header comment of Winery-Strata's
``include/strata/core/layer.hpp``; composition in ``src/core/layer.cpp``,
gdn_layer steps 3-7). The cases are chosen so that a plausible slip (a
dropped decay, a wrong sign in the delta, a transposed state, the pre-update
state in the readout, the wrong head map, SiLU where sigmoid belongs, a norm
on v, a missing q scale, a shifted conv tap) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------ constants --
def test_geometry_matches_pages():
    vals = {}
    with open(os.path.join(GOLDEN, "geometry.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, val = line.split()[:2]
            vals[key] = float(val)
    assert vals["head_dim"] == O.HEAD_DIM
    assert vals["k_heads"] == O.K_HEADS
    assert vals["v_heads"] == O.V_HEADS
    assert vals["conv_channels"] == O.CONV_CHANNELS
    assert vals["q_offset"] == O.Q_OFFSET
    assert vals["k_offset"] == O.K_OFFSET
    assert vals["v_offset"] == O.V_OFFSET
    assert vals["d_conv"] == O.D_CONV
    assert vals["rms_eps"] == O.EPS
    assert O.VALUE_DIM == 6144 == O.V_HEADS * O.HEAD_DIM
    assert O.V_OFFSET + O.VALUE_DIM == O.CONV_CHANNELS


# ------------------------------------------------------ scalar functions --
def test_sigmoid_silu_softplus_closed_forms():
    xs = np.array([-80.0, -30.0, -3.5, -1.0, -1e-3, 0.0, 1e-3, 0.5, 2.0, 30.0, 80.0])
    for x, s, si, sp in zip(xs, O.sigmoid(xs), O.silu(xs), O.softplus(xs)):
        assert s == pytest.approx(1.0 / (1.0 + math.exp(-x)), rel=1e-15, abs=1e-300)
        assert si == pytest.approx(x / (1.0 + math.exp(-x)), rel=1e-15, abs=1e-300)
        ref = math.log1p(math.exp(x)) if x < 30 else x + math.log1p(math.exp(-x))
        assert sp == pytest.approx(ref, rel=1e-15, abs=1e-300)
    assert O.sigmoid(0.0) == 0.5
    assert O.silu(0.0) == 0.0
    assert O.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16)
    # softplus(x) - softplus(-x) = x for every x
    assert np.allclose(O.softplus(xs) - O.softplus(-xs), xs, rtol=0, atol=1e-13)


def test_gates_closed_form():
    # alpha_raw + dt = 0 gives softplus = ln 2, so decay = 2**ssm_a exactly in real arithmetic.
    ssm_a = np.array([-1.0, -2.0, -4.0, -16.0, -0.25])
    beta, decay = O.gates(np.array([0.5, -1.0, 2.0, 0.0, 3.0]), np.zeros(5),
                          np.array([-0.5, 1.0, -2.0, 0.0, -3.0]), ssm_a)
    assert np.allclose(decay, 2.0 ** ssm_a, rtol=1e-14, atol=0)
    assert np.all(beta == 0.5)
    # large beta_raw -> beta -> 1; decay is always in (0, 1] for ssm_a < 0
    beta, decay = O.gates(np.array([40.0]), np.array([40.0]), np.array([0.0]), np.array([-3.0]))
    assert beta[0] == pytest.approx(1.0, abs=1e-15)
    assert decay[0] == pytest.approx(math.exp(-120.0), rel=1e-13)


# ------------------------------------------------------------- the conv --
def test_conv_taps_oldest_first_and_no_bias():
    r = _rng(1)
    C = 64
    hist = r.standard_normal((C, 3)).astype(np.float32)
    x = r.standard_normal(C).astype(np.float32)
    for tap in range(4):
        w = np.zeros((C, 4), np.float32)
        w[:, tap] = 1.0
        xc = O.causal_conv(x, hist, w)
        expect = x if tap == 3 else hist[:, tap]
        assert np.array_equal(xc, expect.astype(np.float64))
    # zero weights -> zero output (no bias term)
    assert np.all(O.causal_conv(x, hist, np.zeros((C, 4), np.float32)) == 0.0)


def test_conv_matches_scalar_loop():
    r = _rng(2)
    C = 32
    hist = r.standard_normal((C, 3)).astype(np.float32)
    x = r.standard_normal(C).astype(np.float32)
    w = r.standard_normal((C, 4)).astype(np.float32)
    xc = O.causal_conv(x, hist, w)
    for c in range(C):
        seq = [float(hist[c, 0]), float(hist[c, 1]), float(hist[c, 2]), float(x[c])]
        exact = sum(Fraction(float(w[c, j])) * Fraction(seq[j]) for j in range(4))
        assert xc[c] == pytest.approx(float(exact), rel=1e-15, abs=1e-15)


def test_conv_state_roll_is_exact_shift():
    r = _rng(3)
    C = 40
    hist = r.standard_normal((C, 3)).astype(np.float32)
    x = r.standard_normal(C).astype(np.float32)
    new = O.roll_conv_state(hist, x)
    assert new.dtype == np.float32
    for c in range(C):
        assert new[c, 0] == hist[c, 1]
        assert new[c, 1] == hist[c, 2]
        assert new[c, 2] == x[c]


# ------------------------------------------------------------ the norms --
def test_l2_normalize_and_q_scale():
    r = _rng(4)
    x = r.standard_normal((5, 128))
    n = O.l2_normalize(x)
    for row, nrow in zip(x, n):
        ss = math.fsum(float(a) * float(a) for a in row)
        expect_norm = math.sqrt(ss / (ss + O.EPS))
        assert math.sqrt(math.fsum(float(a) * float(a) for a in nrow)) == pytest.approx(expect_norm, rel=1e-14)
    # the zero vector stays zero (eps guards the division)
    assert np.all(O.l2_normalize(np.zeros((1, 128))) == 0.0)


def test_preprocess_norms_q_k_not_v_and_scales_q():
    r = _rng(5)
    C = O.CONV_CHANNELS
    x = r.standard_normal(C).astype(np.float32)
    hist = r.standard_normal((C, 3)).astype(np.float32)
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0                          # conv output = x
    p = O.preprocess_token(x, hist, w, np.zeros(48), np.zeros(48), np.zeros(48), -np.ones(48))
    # v is SiLU(x) on its channels, element by element, and NOT normalised
    for c in range(0, O.VALUE_DIM, 97):
        xv = float(x[O.V_OFFSET + c])
        assert p["v"].reshape(-1)[c] == pytest.approx(xv / (1.0 + math.exp(-xv)), rel=1e-15, abs=1e-300)
    vnorm = np.linalg.norm(p["v"], axis=1)
    assert not np.allclose(vnorm, 1.0, atol=0.05)
    # |q| = 1/sqrt(128) (up to eps) and |k| = 1, each computed with fsum from SiLU(x)
    for hk in range(O.K_HEADS):
        for off, got, scale in ((O.Q_OFFSET, p["q"][hk], 1.0 / math.sqrt(128.0)), (O.K_OFFSET, p["k"][hk], 1.0)):
            raw = [float(a) / (1.0 + math.exp(-float(a))) for a in x[off + 128 * hk: off + 128 * (hk + 1)]]
            ss = math.fsum(a * a for a in raw)
            inv = 1.0 / math.sqrt(ss + O.EPS) * scale
            for i in (0, 17, 127):
                assert got[i] == pytest.approx(raw[i] * inv, rel=1e-14)
    # SiLU applies to the whole conv output before the split: q channels too
    assert np.all(p["q"][p["q"] != 0] * np.sign(p["q"][p["q"] != 0]) > 0)


# ----------------------------------------------------- the delta rule ----
def _frac_step(S, k, q, v, beta, decay):
    """The affine form S' = decay (I - beta k k^T) S + beta k v^T and o = S'^T q, in exact rationals."""
    dk, dv = len(S), len(S[0])
    P = [[(Fraction(1) if a == b else Fraction(0)) - beta * k[a] * k[b] for b in range(dk)] for a in range(dk)]
    Sn = [[decay * sum(P[a][c] * S[c][j] for c in range(dk)) + beta * k[a] * v[j] for j in range(dv)]
          for a in range(dk)]
    o = [sum(Sn[a][j] * q[a] for a in range(dk)) for j in range(dv)]
    return Sn, o


@pytest.mark.parametrize("dk,dv,seed", [(2, 4, 0), (3, 2, 1), (4, 4, 2)])
def test_delta_step_matches_affine_form_exactly(dk, dv, seed):
    r = _rng(10 + seed)
    # small dyadic rationals so the fp64 oracle's result is exact or nearly so
    S = (r.integers(-8, 9, size=(dk, dv)) / 8.0)
    k = r.integers(-4, 5, size=dk) / 4.0
    q = r.integers(-4, 5, size=dk) / 4.0
    v = r.integers(-4, 5, size=dv) / 4.0
    beta, decay = 0.75, 0.5
    Sn, o = O.delta_rule_step(S, k, q, v, beta, decay)
    F = lambda a: Fraction(float(a))  # noqa: E731
    Sf, of = _frac_step([[F(a) for a in row] for row in S], [F(a) for a in k], [F(a) for a in q],
                        [F(a) for a in v], F(beta), F(decay))
    assert Sn.shape == (dk, dv) and o.shape == (dv,)
    for a in range(dk):
        for j in range(dv):
            assert Sn[a, j] == float(Sf[a][j])
    for j in range(dv):
        assert o[j] == float(of[j])


def test_delta_step_beta0_decay1_leaves_state_and_reads_out():
    r = _rng(20)
    S = r.standard_normal((128, 128)) * 0.05
    k = O.l2_normalize(r.standard_normal(128))
    q = O.l2_normalize(r.standard_normal(128)) / math.sqrt(128)
    v = r.standard_normal(128)
    Sn, o = O.delta_rule_step(S, k, q, v, 0.0, 1.0)
    assert np.array_equal(Sn, S)
    for j in (0, 5, 64, 127):
        assert o[j] == pytest.approx(math.fsum(S[i, j] * q[i] for i in range(128)), rel=1e-12, abs=1e-15)


def test_delta_step_beta1_unit_k_writes_v():
    r = _rng(21)
    S = r.standard_normal((128, 128)) * 0.05
    k = r.standard_normal(128)
    k /= np.linalg.norm(k)
    v = r.standard_normal(128)
    for decay in (1.0, 0.3):
        Sn, o = O.delta_rule_step(S, k, k, v, 1.0, decay)
        # S'^T k = v exactly in real arithmetic; the readout with q = k is therefore v
        assert np.allclose(Sn.T @ k, v, rtol=0, atol=1e-13)
        assert np.allclose(o, v, rtol=0, atol=1e-13)
        # directions orthogonal to k only decay
        u = r.standard_normal(128)
        u -= (u @ k) * k
        assert np.allclose(Sn.T @ u, decay * (S.T @ u), rtol=0, atol=1e-13)


def test_delta_step_decay0_forgets_state():
    r = _rng(22)
    S = r.standard_normal((128, 128))
    k = r.standard_normal(128)
    q = r.standard_normal(128)
    v = r.standard_normal(128)
    Sn, o = O.delta_rule_step(S, k, q, v, 1.0, 0.0)
    assert np.array_equal(Sn, np.outer(k, v))
    for j in (0, 77):
        assert o[j] == pytest.approx(v[j] * math.fsum(k[i] * q[i] for i in range(128)), rel=1e-13)


def test_delta_step_readout_uses_updated_state():
    # with beta = 1, unit k and q = k, the updated state reads out v; the old one would not
    r = _rng(23)
    S = r.standard_normal((128, 128))
    k = r.standard_normal(128)
    k /= np.linalg.norm(k)
    v = np.zeros(128)
    _, o = O.delta_rule_step(S, k, k, v, 1.0, 1.0)
    assert np.max(np.abs(o)) < 1e-12
    assert np.max(np.abs(S.T @ k)) > 0.1


# ------------------------------------------------------ the output norm --
def test_gated_rms_norm_closed_forms():
    r = _rng(30)
    w = r.standard_normal(128)
    o = np.full(128, 3.0)
    z = np.zeros(128)
    y = O.gated_rms_norm(o, z, w)
    # constant o: rms = sqrt(9 + eps); sigmoid(0) = 1/2 (SiLU(0) would give 0)
    assert np.allclose(y, 3.0 / math.sqrt(9.0 + O.EPS) * w * 0.5, rtol=1e-15, atol=0)
    assert np.all(O.gated_rms_norm(np.zeros(128), z, w) == 0.0)
    o = r.standard_normal(128)
    z = r.standard_normal(128)
    y = O.gated_rms_norm(o, z, w)
    ms = math.fsum(a * a for a in o) / 128
    for j in (0, 63, 127):
        assert y[j] == pytest.approx(o[j] / math.sqrt(ms + O.EPS) * w[j] / (1 + math.exp(-z[j])), rel=1e-14)
    ys = O.gated_rms_norm(o, z, w, gate="silu")
    assert ys[5] == pytest.approx(o[5] / math.sqrt(ms + O.EPS) * w[5] * z[5] / (1 + math.exp(-z[5])), rel=1e-14)


def test_gated_rms_norm_silu_variant_closed_forms():
    """The SiLU-gated variant (the earlier model's output gate, named beside the sigmoid in the
    header comment of include/strata/core/layer.hpp): SiLU(0) = 0 exactly, SiLU(z) -> z for large z
    and -> 0 from below for very negative z. Sigmoid would give w/2, w and 0+ there instead."""
    r = _rng(31)
    w = r.standard_normal(128)
    o = np.full(128, 3.0)
    unit = 3.0 / math.sqrt(9.0 + O.EPS)  # o / rms(o) for a constant o = 3
    assert np.all(O.gated_rms_norm(o, np.zeros(128), w, gate="silu") == 0.0)
    y = O.gated_rms_norm(o, np.full(128, 40.0), w, gate="silu")
    # SiLU(40) = 40 / (1 + e^-40) = 40 (1 - 4.2e-18 ...): equal to 40 in fp64 within one ulp
    assert np.allclose(y, unit * w * 40.0, rtol=2e-16, atol=0)
    y = O.gated_rms_norm(o, np.full(128, -40.0), w, gate="silu")
    # SiLU(-40) = -40 e^-40 / (1 + e^-40): a tiny value of the opposite sign to w
    assert np.allclose(y, -unit * w * 40.0 * math.exp(-40.0), rtol=1e-14, atol=0)
    assert np.all(np.sign(y) == -np.sign(w))


# ------------------------------------------------------- the whole step --
def _one_layer_inputs(seed, T=1, zero_state=False):
    r = _rng(seed)
    C, V = O.CONV_CHANNELS, O.VALUE_DIM
    sl = {
        "qkv": r.standard_normal((T, C)).astype(np.float32),
        "z": r.standard_normal((T, V)).astype(np.float32),
        "alpha": r.standard_normal((T, 48)).astype(np.float32),
        "beta": r.standard_normal((T, 48)).astype(np.float32),
        "conv_state": r.standard_normal((C, 3)).astype(np.float32),
        "state": (np.zeros((48, 128, 128)) if zero_state else r.standard_normal((48, 128, 128)) * 0.05
                  ).astype(np.float32),
    }
    wts = {
        "dt": (r.standard_normal(48) * 0.5).astype(np.float32),
        "ssm_a": (-np.exp(r.random(48) * math.log(16))).astype(np.float32),
        "conv_w": (r.standard_normal((C, 4)) * 0.25).astype(np.float32),
        "ssm_norm": (1 + 0.1 * r.standard_normal(128)).astype(np.float32),
    }
    return sl, wts


def test_zero_state_one_step_closed_form():
    """From S = 0: S' = beta k v^T, o = beta (k.q) v, so y = c v / sqrt(c^2 mean(v^2) + eps) * w * sigmoid(z)."""
    sl, wts = _one_layer_inputs(40, zero_state=True)
    wts["conv_w"][:] = 0.0
    wts["conv_w"][:, 3] = 1.0                      # conv output = x
    y, st, cs = O.gdn_decode_slice(sl, wts)
    x = [float(a) for a in sl["qkv"][0]]
    h = [a / (1.0 + math.exp(-a)) for a in x]
    for hv in (0, 1, 2, 3, 25, 47):
        hk = hv // 3
        qr = h[128 * hk: 128 * hk + 128]
        kr = h[2048 + 128 * hk: 2048 + 128 * hk + 128]
        vv = h[4096 + 128 * hv: 4096 + 128 * hv + 128]
        qn = math.sqrt(math.fsum(a * a for a in qr) + O.EPS)
        kn = math.sqrt(math.fsum(a * a for a in kr) + O.EPS)
        kq = math.fsum((a / kn) * (b / qn / math.sqrt(128)) for a, b in zip(kr, qr))
        bta = 1.0 / (1.0 + math.exp(-float(sl["beta"][0, hv])))
        c = bta * kq
        mv = math.fsum(a * a for a in vv) / 128
        for j in (0, 31, 127):
            zz = float(sl["z"][0, 128 * hv + j])
            expect = c * vv[j] / math.sqrt(c * c * mv + O.EPS) * float(wts["ssm_norm"][j]) / (1 + math.exp(-zz))
            assert y[0, 128 * hv + j] == pytest.approx(expect, rel=1e-11, abs=1e-14)
            # state column j = beta * k * v_j
            assert st[hv, 7, j] == pytest.approx(bta * kr[7] / kn * vv[j], rel=1e-12, abs=1e-16)


def test_head_map_v_head_reads_k_head_div_3():
    sl, wts = _one_layer_inputs(41, zero_state=True)
    wts["conv_w"][:] = 0.0
    wts["conv_w"][:, 3] = 1.0
    # zero every q/k head except k-head 5 -> only v heads 15, 16, 17 get a nonzero update
    sl["qkv"][0, :4096] = 0.0
    sl["qkv"][0, 128 * 5: 128 * 6] = 1.0
    sl["qkv"][0, 2048 + 128 * 5: 2048 + 128 * 6] = np.linspace(-1, 1, 128)
    _, st, _ = O.gdn_decode_slice(sl, wts)
    touched = [h for h in range(48) if np.any(st[h] != 0.0)]
    assert touched == [15, 16, 17]
    assert [O.v_head_to_k_head(h) for h in (0, 2, 3, 47)] == [0, 0, 1, 15]


def test_t_steps_equal_single_steps_and_ragged_prefix():
    sl, wts = _one_layer_inputs(42, T=4)
    y4, st4, cs4 = O.gdn_decode_slice(sl, wts)
    st = sl["state"]
    cs = sl["conv_state"]
    for t in range(4):
        one = {k: (v[t:t + 1] if k in ("qkv", "z", "alpha", "beta") else v) for k, v in sl.items()}
        one["state"], one["conv_state"] = st, cs
        y1, st, cs = O.gdn_decode_slice(one, wts)
        assert np.array_equal(y1[0], y4[t])
    assert np.array_equal(st, st4) and np.array_equal(cs, cs4)
    # ragged: n = 2 equals a T = 2 call on the prefix, and leaves later y as NaN
    y2, st2, cs2 = O.gdn_decode_slice(sl, wts, n=2)
    pre = {k: (v[:2] if k in ("qkv", "z", "alpha", "beta") else v) for k, v in sl.items()}
    yp, stp, csp = O.gdn_decode_slice(pre, wts)
    assert np.array_equal(y2[:2], yp) and np.all(np.isnan(y2[2:]))
    assert np.array_equal(st2, stp) and np.array_equal(cs2, csp)
    # n = 0 changes nothing
    y0, st0, cs0 = O.gdn_decode_slice(sl, wts, n=0)
    assert np.all(np.isnan(y0)) and np.array_equal(st0, sl["state"]) and np.array_equal(cs0, sl["conv_state"])


def test_conv_history_after_t_tokens():
    sl, wts = _one_layer_inputs(43, T=5)
    _, _, cs = O.gdn_decode_slice(sl, wts, n=2)
    # after two tokens: (old[2], x0, x1)
    assert np.array_equal(cs[:, 0], sl["conv_state"][:, 2])
    assert np.array_equal(cs[:, 1], sl["qkv"][0])
    assert np.array_equal(cs[:, 2], sl["qkv"][1])
    _, _, cs = O.gdn_decode_slice(sl, wts)
    assert np.array_equal(cs, sl["qkv"][2:5].T)


def test_batch_permutation_equivariance():
    r = _rng(44)
    B, L, T = 3, 2, 2
    sls = [[_one_layer_inputs(100 + 10 * b + l, T=T)[0] for l in range(L)] for b in range(B)]
    wl = [_one_layer_inputs(200 + l)[1] for l in range(L)]
    stack = lambda key: np.stack([np.stack([sls[b][l][key] for l in range(L)]) for b in range(B)])  # noqa: E731
    wst = lambda key: np.stack([wl[l][key] for l in range(L)])  # noqa: E731
    args = [stack("qkv"), stack("z"), stack("alpha"), stack("beta"), wst("dt"), wst("ssm_a"), wst("conv_w"),
            wst("ssm_norm"), stack("conv_state"), stack("state")]
    lens = np.array([2, 1, 2])
    y, st, cs = O.gdn_decode(*args, seq_len=lens)
    perm = r.permutation(B)
    pargs = [a[perm] if a.shape[0] == B and i not in (4, 5, 6, 7) else a for i, a in enumerate(args)]
    yp, stp, csp = O.gdn_decode(*pargs, seq_len=lens[perm])
    assert np.array_equal(np.isnan(yp), np.isnan(y[perm]))
    assert np.array_equal(np.nan_to_num(yp), np.nan_to_num(y[perm]))
    assert np.array_equal(stp, st[perm]) and np.array_equal(csp, cs[perm])


# ------------------------------------------- the alpha/beta projection --
def test_ab_gates_one_hot_input_picks_a_weight_column():
    r = _rng(50)
    E = 64
    wa = r.standard_normal((48, E))
    wb = r.standard_normal((48, E))
    dt = r.standard_normal(48)
    ssm_a = -np.exp(r.random(48))
    x = np.zeros(E)
    x[17] = 1.0
    gate, beta = O.ab_gates(x, wa, wb, dt, ssm_a)
    for h in (0, 20, 47):
        a = wa[h, 17] + dt[h]
        assert gate[h] == pytest.approx((max(a, 0) + math.log1p(math.exp(-abs(a)))) * ssm_a[h], rel=1e-14)
        assert beta[h] == pytest.approx(1.0 / (1.0 + math.exp(-wb[h, 17])), rel=1e-14)


def test_ab_gates_matches_scalar_sums_and_feeds_the_step():
    r = _rng(51)
    E = 96
    x = r.standard_normal((3, E))
    wa = r.standard_normal((48, E)) / math.sqrt(E)
    wb = r.standard_normal((48, E)) / math.sqrt(E)
    dt = r.standard_normal(48) * 0.5
    ssm_a = -np.exp(r.random(48) * math.log(16))
    gate, beta = O.ab_gates(x, wa, wb, dt, ssm_a)
    assert gate.shape == (3, 48) and beta.shape == (3, 48)
    for i, h in ((0, 0), (1, 33), (2, 47)):
        ar = math.fsum(x[i, k] * wa[h, k] for k in range(E))
        br = math.fsum(x[i, k] * wb[h, k] for k in range(E))
        assert gate[i, h] == pytest.approx(O.softplus(ar + dt[h]) * ssm_a[h], rel=1e-12)
        assert beta[i, h] == pytest.approx(1.0 / (1.0 + math.exp(-br)), rel=1e-12)
    # the step fed with (log decay, beta) equals the step fed with the raw projections
    sl, wts = _one_layer_inputs(52)
    ar = (x[:1] @ wa.T).astype(np.float64)
    br = (x[:1] @ wb.T).astype(np.float64)
    raw = dict(sl, alpha=ar, beta=br)
    wts = dict(wts, dt=dt, ssm_a=ssm_a)
    y1, s1, _ = O.gdn_decode_slice(raw, wts)
    g1, b1 = O.ab_gates(x[:1], wa, wb, dt, ssm_a)
    y2, s2, _ = O.gdn_decode_slice(dict(sl, alpha=g1, beta=b1), wts, gates_ready=True)
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-14) and np.allclose(s1, s2, rtol=1e-12, atol=1e-16)


# ------------------------------------------------ the input projections --
def test_in_proj_one_hot_rows_select_and_scale_inputs():
    """A weight row with one non-zero entry c picks x[c] times that entry: exact for
    power-of-two entries, whatever the row order."""
    r = _rng(60)
    E = 40
    x = r.standard_normal((2, E)).astype(np.float32)
    cols_q, cols_g = r.permutation(E)[:9], r.permutation(E)[:5]
    sq = np.array([1.0, -0.5, 0.125, 2.0, -1.0, 4.0, 0.25, -8.0, 1.0])
    sg = np.array([-1.0, 0.5, 16.0, -0.0625, 1.0])
    wq = np.zeros((9, E))
    wq[np.arange(9), cols_q] = sq
    wg = np.zeros((5, E))
    wg[np.arange(5), cols_g] = sg
    qkv, z = O.in_proj(x, wq, wg)
    assert qkv.shape == (2, 9) and z.shape == (2, 5)
    assert np.array_equal(qkv, x[:, cols_q].astype(np.float64) * sq)
    assert np.array_equal(z, x[:, cols_g].astype(np.float64) * sg)


def test_in_proj_equals_exact_rational_sums():
    """On small dyadic inputs every product and partial sum is exact in float64, so the
    projection must equal the rational dot product of each weight row with x exactly."""
    from fractions import Fraction

    r = _rng(61)
    E, NQ, NZ, M = 11, 7, 4, 3
    x = r.integers(-64, 64, (M, E)) / 16.0
    wq = r.integers(-128, 128, (NQ, E)) / 64.0
    wg = r.integers(-128, 128, (NZ, E)) / 64.0
    qkv, z = O.in_proj(x, wq, wg)
    assert qkv.shape == (M, NQ) and z.shape == (M, NZ)
    for m in range(M):
        for c in range(NQ):
            assert qkv[m, c] == float(sum(Fraction(x[m, k]) * Fraction(wq[c, k]) for k in range(E)))
        for c in range(NZ):
            assert z[m, c] == float(sum(Fraction(x[m, k]) * Fraction(wg[c, k]) for k in range(E)))
