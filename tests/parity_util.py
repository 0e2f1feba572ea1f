"""Helpers shared by the GPU parity tests: inputs on the device, the oracle on
sampled slices, and the error measures with the tolerance in one place.

Tolerance. A result matches the oracle when, for every slice, the normwise
relative error ``max |gpu - oracle| / max |oracle|`` is at most 1e-4 (y per
(sequence, layer, token) 6144-vector; state per (sequence, layer, v-head)
128x128 tile). conv_state must be bit-identical.

The element-wise relative error ``|gpu - oracle| / max(|oracle|, 1e-3 max |oracle|)``
per slice is reported beside it (``elementwise_error``); it is not a pass
criterion. A normwise error e bounds it by 1000 e.
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


def elementwise_error(g: np.ndarray, r: np.ndarray, rows: int) -> float:
    """Worst element-wise relative error over slices of ``rows`` elements, with the
    denominator floored at 1e-3 of the slice's largest reference magnitude; NaN
    (invalid) slices of the reference are skipped."""
    a = np.asarray(g, np.float64).reshape(-1, rows)
    b = np.asarray(r, np.float64).reshape(-1, rows)
    keep = ~np.isnan(b[:, 0])
    a, b = a[keep], b[keep]
    if a.size == 0:
        return 0.0
    floor = 1e-3 * np.abs(b).max(axis=1, keepdims=True)
    den = np.maximum(np.abs(b), np.where(floor > 0, floor, 1.0))
    return float(np.max(np.abs(a - b) / den))


def report(label: str, gy, ry, gs, rs) -> str:
    """One line with the normwise and element-wise errors of y and the state."""
    return (f"{label}: y normwise {y_errors(gy, ry):.2e} element-wise {elementwise_error(gy, ry, ry.shape[-1]):.2e}; "
            f"state normwise {state_errors(gs, rs):.2e} element-wise {elementwise_error(gs, rs, 128 * 128):.2e}")


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
