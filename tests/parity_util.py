"""Helpers shared by the GPU parity tests: inputs on the device, the oracle on
sampled slices, and the error measures with the tolerance in one place.

Tolerance. A result matches the oracle when, for every slice, the normwise
relative error ``max |gpu - oracle| / max |oracle|`` is at most 1e-4 (y per
(sequence, layer, token) 6144-vector; state per (sequence, layer, v-head)
128x128 tile). conv_state must be bit-identical.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

TOL = 1e-4


def to_device(h: dict, dev) -> dict:
    return {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev)) for k, v in h.items()}


def run_step(g, t: dict, y=None, seq_len="auto", flags=None):
    """Runs one decode call on device tensors ``t`` (updated in place); returns y."""
    if y is None:
        y = torch.full(t["z"].shape, float("nan"), device=t["z"].device)
    sl = t.get("seq_len") if seq_len == "auto" else seq_len
    args = (t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
            t["conv_state"], t["state"], y)
    if flags is not None:
        g.gdn_decode_step_ex(*args, seq_len=sl, flags=flags)
    elif sl is None:
        g.gdn_decode_step(*args)
    else:
        g.gdn_decode_step_varlen(*args, sl)
    return y


def y_errors(gy: np.ndarray, ry: np.ndarray) -> float:
    """Worst normwise error over the (.., t) rows of y; NaN rows (invalid tokens) must coincide."""
    assert np.array_equal(np.isnan(gy), np.isnan(ry)), "y written where it must not be (or missing)"
    worst = 0.0
    rows_g = gy.reshape(-1, gy.shape[-1])
    rows_r = ry.reshape(-1, ry.shape[-1])
    for a, b in zip(rows_g, rows_r):
        if np.isnan(b[0]):
            continue
        den = np.abs(b).max()
        worst = max(worst, np.abs(a - b).max() / den if den > 0 else np.abs(a).max())
    return worst


def state_errors(gs: np.ndarray, rs: np.ndarray) -> float:
    """Worst normwise error over the 128x128 tiles of a state."""
    a = gs.reshape(-1, 128 * 128).astype(np.float64)
    b = rs.reshape(-1, 128 * 128)
    den = np.abs(b).max(axis=1)
    num = np.abs(a - b).max(axis=1)
    return float(np.max(np.where(den > 0, num / np.where(den > 0, den, 1), num)))


def oracle_full(h: dict, gate="sigmoid"):
    return oracle.gdn_decode(h["qkv"], h["z"], h["alpha"], h["beta"], h["dt"], h["ssm_a"], h["conv_w"],
                             h["ssm_norm"], h["conv_state"], h["state"], seq_len=h["seq_len"], gate=gate)


def oracle_slice(w: W.Workload, b: int, l: int):
    """The oracle on one (sequence, layer) slice, regenerated from the workload's seed."""
    sl = W.sequence_slice(w, b, l)
    wts = W.layer_weights(w, l)
    lens = W.seq_lens(w)
    n = None if lens is None else int(lens[b])
    return oracle.gdn_decode_slice(sl, wts, n)
