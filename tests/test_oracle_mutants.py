"""The pins are strong enough: each plausible slip, planted in the oracle on the
CPU, makes at least one pin of ``test_oracle_pins.py`` fail."""
import math

import numpy as np
import pytest

import oracle as O
import tests.test_oracle_pins as P

PINS = [getattr(P, n) for n in dir(P) if n.startswith("test_") and callable(getattr(P, n))]


def _run_pins():
    failures = 0
    for fn in PINS:
        try:
            if fn is P.test_delta_step_matches_affine_form_exactly:
                for args in [(2, 4, 0), (3, 2, 1)]:
                    fn(*args)
            else:
                fn()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


def _step_no_decay(S, k, q, v, beta, decay):
    S = np.asarray(S, np.float64)
    kv = S.T @ k
    d = (v - kv) * beta
    S = S + np.outer(k, d)
    return S, S.T @ q


def _step_sign(S, k, q, v, beta, decay):
    S = np.asarray(S, np.float64) * decay
    kv = S.T @ k
    d = (kv - v) * beta
    S = S + np.outer(k, d)
    return S, S.T @ q


def _step_transposed(S, k, q, v, beta, decay):
    S = np.asarray(S, np.float64) * decay
    kv = S @ np.resize(k, S.shape[1])
    d = (v - kv) * beta
    S = S + np.outer(k, d)
    return S, S.T @ q


def _step_old_readout(S, k, q, v, beta, decay):
    S = np.asarray(S, np.float64) * decay
    kv = S.T @ k
    o = S.T @ q
    d = (v - kv) * beta
    return S + np.outer(k, d), o


def _step_decay_after(S, k, q, v, beta, decay):
    S = np.asarray(S, np.float64)
    kv = S.T @ k
    d = (v - kv) * beta
    S = (S + np.outer(k, d)) * decay
    return S, S.T @ q


def _norm_silu_gate(o, z, w, eps=O.EPS, gate="sigmoid"):
    o = np.asarray(o, np.float64)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * w * O.silu(z)


def _norm_sigmoid_always(o, z, w, eps=O.EPS, gate="sigmoid"):
    o = np.asarray(o, np.float64)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * w * O.sigmoid(z)


def _norm_sum(o, z, w, eps=O.EPS, gate="sigmoid"):
    o = np.asarray(o, np.float64)
    return o / np.sqrt(np.sum(o * o, axis=-1, keepdims=True) + eps) * w * O.sigmoid(z)


def _l2_eps_outside(x, eps=O.EPS):
    x = np.asarray(x, np.float64)
    return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)


def _conv_reversed(x, conv_state, conv_w):
    hist = np.asarray(conv_state, np.float64)
    w = np.asarray(conv_w, np.float64)
    return w[:, 3] * hist[:, 0] + w[:, 2] * hist[:, 1] + w[:, 1] * hist[:, 2] + w[:, 0] * np.asarray(x, np.float64)


def _roll_wrong(conv_state, x):
    hist = np.asarray(conv_state, np.float32)
    out = hist.copy()
    out[:, 0] = np.asarray(x, np.float32)
    return out


def _softplus_wrong(x):
    return np.log(np.exp(np.asarray(x, np.float64)))


def _make_pre(normalize_v=False, scale_q=True, silu_qk_only=False):
    orig = O.preprocess_token

    def pre(x, conv_state, conv_w, alpha_raw, beta_raw, dt, ssm_a, gates_ready=False):
        p = orig(x, conv_state, conv_w, alpha_raw, beta_raw, dt, ssm_a, gates_ready)
        if normalize_v:
            p["v"] = O.l2_normalize(p["v"])
        if not scale_q:
            p["q"] = p["q"] * math.sqrt(O.HEAD_DIM)
        if silu_qk_only:
            p["v"] = p["xc"][O.V_OFFSET:].reshape(O.V_HEADS, O.HEAD_DIM)
        return p

    return pre


def _proj_drop_last(x, w_qkv, w_gate):
    x = np.asarray(x, np.float64)
    return x[..., :-1] @ np.asarray(w_qkv)[:, :-1].T, x[..., :-1] @ np.asarray(w_gate)[:, :-1].T


def _proj_rows_shifted(x, w_qkv, w_gate):
    x = np.asarray(x, np.float64)
    return x @ np.roll(np.asarray(w_qkv), 1, axis=0).T, x @ np.roll(np.asarray(w_gate), 1, axis=0).T


def _proj_swapped(x, w_qkv, w_gate):
    x = np.asarray(x, np.float64)
    return x @ np.asarray(w_gate).T, x @ np.asarray(w_qkv).T


MUTANTS = {
    "no decay": ("delta_rule_step", _step_no_decay),
    "sign of delta": ("delta_rule_step", _step_sign),
    "transposed state": ("delta_rule_step", _step_transposed),
    "readout before update": ("delta_rule_step", _step_old_readout),
    "decay after update": ("delta_rule_step", _step_decay_after),
    "head map h % 16": ("v_head_to_k_head", lambda h: h % 16),
    "SiLU output gate": ("gated_rms_norm", _norm_silu_gate),
    "sigmoid for SiLU in the gate variant": ("gated_rms_norm", _norm_sigmoid_always),
    "RMS with sum": ("gated_rms_norm", _norm_sum),
    "eps outside sqrt": ("l2_normalize", _l2_eps_outside),
    "conv taps reversed": ("causal_conv", _conv_reversed),
    "conv roll wrong": ("roll_conv_state", _roll_wrong),
    "softplus dropped log1p": ("softplus", _softplus_wrong),
    "v normalised": ("preprocess_token", None),
    "q not scaled": ("preprocess_token", None),
    "SiLU after split": ("preprocess_token", None),
    "projection drops an input": ("in_proj", _proj_drop_last),
    "projection rows shifted": ("in_proj", _proj_rows_shifted),
    "projections swapped": ("in_proj", _proj_swapped),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    if fn is None:
        fn = _make_pre(normalize_v=name == "v normalised", scale_q=name != "q not scaled",
                       silu_qk_only=name == "SiLU after split")
    monkeypatch.setattr(O, attr, fn)
    assert _run_pins() >= 1, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins() == 0
