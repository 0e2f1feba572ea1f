"""Seeded synthetic workloads for the Gated DeltaNet (GDN) decode step.

This module generates inputs and nothing else: it holds none of the step's
arithmetic. The fp64 oracle (under ``oracle/``), the CUDA library's tests and
``bench.py`` all draw their inputs from here, so both sides of every parity
check see the same bytes.

Every tensor slice is produced by its own Philox4x32-10 stream (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC'11, as implemented by
``numpy.random.Philox``), keyed by ``(seed, tensor id, b, l)``. Any single
(sequence, layer) slice can therefore be regenerated on its own, which lets
the oracle check sampled slices of a 14.5 GB workload without holding it.

Distributions (the second parameter of N(mu, sigma) is a standard deviation):

==============  =====================================================
qkv, z          N(0, 1) per token
alpha_raw       N(0, 1); N(-2, 1) in the large-batch workload
beta_raw        N(0, 1); N(2, 1) in the large-batch workload
dt              N(0, 0.5) per layer and v-head
ssm_a           -exp(U(0, ln 16)) per layer and v-head (so ssm_a < 0)
conv_w          N(0, 0.25), [C][4] per layer
ssm_norm        N(1, 0.1), [128] per layer
conv_state      N(0, 1), [C][3] per (sequence, layer)
state           N(0, 0.05), [48][128][128] per (sequence, layer);
                zeros in the 64-step single-sequence workload
seq_len         U{1..T} per sequence in the ragged verify workload
==============  =====================================================
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

# Shapes of the fixed geometry (head dim, heads, channel split). These are the
# tensor shapes the workloads are drawn in, not arithmetic of the step.
HEAD_DIM = 128
K_HEADS = 16
V_HEADS = 48
CONV_CHANNELS = 10240
VALUE_DIM = 6144
D_CONV = 4
N_EMBD = 2560  # model width feeding the alpha/beta projections (their rows hold 2,560 elements)

# Tensor ids mixed into every Philox key.
_TID = {
    "qkv": 1, "z": 2, "alpha": 3, "beta": 4, "dt": 5, "ssm_a": 6,
    "conv_w": 7, "ssm_norm": 8, "conv_state": 9, "state": 10, "seq_len": 11,
    "x": 12, "w_alpha": 13, "w_beta": 14, "w_qkv": 15, "w_gate": 16,
}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: B sequences x L layers x T tokens."""

    name: str
    B: int
    L: int
    T: int
    seed: int
    state_zero: bool = False
    alpha_mean: float = 0.0
    beta_mean: float = 0.0
    ragged: bool = False

    @property
    def updates(self) -> int:
        """State updates (sequence x layer x token) when every step is valid."""
        return self.B * self.L * self.T

    def scaled(self, B: int | None = None, L: int | None = None, T: int | None = None,
               name: str | None = None) -> "Workload":
        """Same recipe and seed with other sizes (for small parity cases)."""
        return Workload(name or self.name, B or self.B, L or self.L, T or self.T, self.seed,
                        self.state_zero, self.alpha_mean, self.beta_mean, self.ragged)


# The five workloads, named for what they are.
WORKLOADS = {
    "decode_b1_l1_t1": Workload("decode_b1_l1_t1", 1, 1, 1, 20260000),
    "decode_b1_l36_t64_zero_state": Workload("decode_b1_l36_t64_zero_state", 1, 36, 64, 20260001,
                                             state_zero=True),
    "decode_b64_l36_t1": Workload("decode_b64_l36_t1", 64, 36, 1, 20260002),
    "decode_b128_l36_t1_beta_hi_decay_hi": Workload("decode_b128_l36_t1_beta_hi_decay_hi", 128, 36, 1,
                                                    20260003, alpha_mean=-2.0, beta_mean=2.0),
    "verify_b16_l36_t8_ragged": Workload("verify_b16_l36_t8_ragged", 16, 36, 8, 20260004, ragged=True),
}


def _rng(seed: int, tensor: str, *idx: int) -> np.random.Generator:
    key = np.random.SeedSequence([seed, _TID[tensor], *idx])
    return np.random.Generator(np.random.Philox(key))


def _normal(seed, tensor, idx, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _rng(seed, tensor, *idx).standard_normal(out=out, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    if mean != 0.0:
        out += np.float32(mean)
    return out


def layer_weights(w: Workload, l: int) -> dict:
    """Per-layer weights shared by every sequence: dt, ssm_a, conv_w, ssm_norm."""
    u = np.empty(V_HEADS, np.float64)
    _rng(w.seed, "ssm_a", l).random(out=u)
    ssm_a = (-np.exp(u * math.log(16.0))).astype(np.float32)
    return {
        "dt": _normal(w.seed, "dt", (l,), (V_HEADS,), std=0.5),
        "ssm_a": ssm_a,
        "conv_w": _normal(w.seed, "conv_w", (l,), (CONV_CHANNELS, D_CONV), std=0.25),
        "ssm_norm": _normal(w.seed, "ssm_norm", (l,), (HEAD_DIM,), mean=1.0, std=0.1),
    }


def sequence_slice(w: Workload, b: int, l: int) -> dict:
    """Per-(sequence, layer) tensors: the T tokens' activations and the two states."""
    T = w.T
    if w.state_zero:
        state = np.zeros((V_HEADS, HEAD_DIM, HEAD_DIM), np.float32)
    else:
        state = _normal(w.seed, "state", (b, l), (V_HEADS, HEAD_DIM, HEAD_DIM), std=0.05)
    return {
        "qkv": _normal(w.seed, "qkv", (b, l), (T, CONV_CHANNELS)),
        "z": _normal(w.seed, "z", (b, l), (T, VALUE_DIM)),
        "alpha": _normal(w.seed, "alpha", (b, l), (T, V_HEADS), mean=w.alpha_mean),
        "beta": _normal(w.seed, "beta", (b, l), (T, V_HEADS), mean=w.beta_mean),
        "conv_state": _normal(w.seed, "conv_state", (b, l), (CONV_CHANNELS, D_CONV - 1)),
        "state": state,
    }


def seq_lens(w: Workload) -> np.ndarray | None:
    """Valid lengths per sequence (int32, in 1..T) for ragged workloads, else None."""
    if not w.ragged:
        return None
    return _rng(w.seed, "seq_len").integers(1, w.T + 1, size=w.B).astype(np.int32)


def host_inputs(w: Workload, threads: int = 8) -> dict:
    """All inputs of a workload as host float32 arrays in the library's layout.

    Layout (outermost first): qkv [B][L][T][C], z [B][L][T][V], alpha/beta
    [B][L][T][48], dt/ssm_a [L][48], conv_w [L][C][4], ssm_norm [L][128],
    conv_state [B][L][C][3], state [B][L][48][128][128]. Meant for workloads
    that fit in host memory comfortably.
    """
    B, L, T = w.B, w.L, w.T
    out = {
        "qkv": np.empty((B, L, T, CONV_CHANNELS), np.float32),
        "z": np.empty((B, L, T, VALUE_DIM), np.float32),
        "alpha": np.empty((B, L, T, V_HEADS), np.float32),
        "beta": np.empty((B, L, T, V_HEADS), np.float32),
        "dt": np.empty((L, V_HEADS), np.float32),
        "ssm_a": np.empty((L, V_HEADS), np.float32),
        "conv_w": np.empty((L, CONV_CHANNELS, D_CONV), np.float32),
        "ssm_norm": np.empty((L, HEAD_DIM), np.float32),
        "conv_state": np.empty((B, L, CONV_CHANNELS, D_CONV - 1), np.float32),
        "state": np.empty((B, L, V_HEADS, HEAD_DIM, HEAD_DIM), np.float32),
    }

    def fill_layer(l):
        for k, v in layer_weights(w, l).items():
            out[k][l] = v

    def fill_seq(bl):
        b, l = divmod(bl, L)
        for k, v in sequence_slice(w, b, l).items():
            out[k][b, l] = v

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(fill_layer, range(L)))
        list(ex.map(fill_seq, range(B * L)))
    out["seq_len"] = seq_lens(w)
    return out


def device_inputs(w: Workload, device, threads: int = 16, batch_rows: tuple | None = None) -> dict:
    """All inputs of a workload as contiguous torch float32 tensors on ``device``.

    Slices are generated on the host (in parallel threads, one Philox stream
    per slice) and copied in, so the bytes equal ``sequence_slice`` /
    ``layer_weights`` for every (b, l). ``batch_rows`` = (b0, b1) generates
    only sequences b0..b1-1 of the workload (used to shard the batch); the
    returned tensors then have B = b1 - b0 rows.
    """
    import torch

    b0, b1 = batch_rows if batch_rows is not None else (0, w.B)
    B, L, T = b1 - b0, w.L, w.T
    f32 = dict(dtype=torch.float32, device=device)
    t = {
        "qkv": torch.empty((B, L, T, CONV_CHANNELS), **f32),
        "z": torch.empty((B, L, T, VALUE_DIM), **f32),
        "alpha": torch.empty((B, L, T, V_HEADS), **f32),
        "beta": torch.empty((B, L, T, V_HEADS), **f32),
        "dt": torch.empty((L, V_HEADS), **f32),
        "ssm_a": torch.empty((L, V_HEADS), **f32),
        "conv_w": torch.empty((L, CONV_CHANNELS, D_CONV), **f32),
        "ssm_norm": torch.empty((L, HEAD_DIM), **f32),
        "conv_state": torch.empty((B, L, CONV_CHANNELS, D_CONV - 1), **f32),
        "state": torch.empty((B, L, V_HEADS, HEAD_DIM, HEAD_DIM), **f32),
    }
    for l in range(L):
        for k, v in layer_weights(w, l).items():
            t[k][l].copy_(torch.from_numpy(v))

    def gen(b):
        return [sequence_slice(w, b, l) for l in range(L)]

    # A bounded window of sequences in flight keeps host memory at O(threads)
    # slices even for the 14.5 GB workload.
    window = 2 * max(1, threads)
    with ThreadPoolExecutor(max(1, threads)) as ex:
        pending = {}
        nxt = b0
        for b in range(b0, b1):
            while nxt < b1 and nxt < b + window:
                pending[nxt] = ex.submit(gen, nxt)
                nxt += 1
            for l, sl in enumerate(pending.pop(b).result()):
                for k, v in sl.items():
                    t[k][b - b0, l].copy_(torch.from_numpy(v))
    lens = seq_lens(w)
    t["seq_len"] = None if lens is None else torch.from_numpy(lens[b0:b1].copy()).to(device)
    return t


# ---------------------------------------------------------------------------
# Inputs of the fused alpha/beta projection: the layer input x ~ N(0, 1) per
# token and BF16 weights ~ N(0, 1/sqrt(n_embd)) (so the raw projections are
# about N(0, 1), like the raw alpha and beta of the decode workloads).
# ---------------------------------------------------------------------------
def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); returns the 16-bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def ab_weights(w: Workload, l: int, n_embd: int = N_EMBD) -> dict:
    """BF16 alpha/beta projection weights of layer l: bit patterns [48][n_embd] and their float32 values."""
    out = {}
    for name in ("w_alpha", "w_beta"):
        bits = to_bf16_bits(_normal(w.seed, name, (l,), (V_HEADS, n_embd), std=1.0 / math.sqrt(n_embd)))
        out[name] = bits
        out[name + "_f32"] = bf16_bits_to_float(bits)
    return out


def ab_x(w: Workload, b: int, l: int, n_embd: int = N_EMBD) -> np.ndarray:
    """The layer input rows [T][n_embd] of (sequence b, layer l)."""
    return _normal(w.seed, "x", (b, l), (w.T, n_embd))


def host_ab_inputs(w: Workload, n_embd: int = N_EMBD) -> dict:
    """x [B][L][T][n_embd], BF16 weights [L][48][n_embd] (bits and float32 values), dt and ssm_a [L][48]."""
    B, L, T = w.B, w.L, w.T
    x = np.empty((B, L, T, n_embd), np.float32)
    for b in range(B):
        for l in range(L):
            x[b, l] = ab_x(w, b, l, n_embd)
    wts = [ab_weights(w, l, n_embd) for l in range(L)]
    lw = [layer_weights(w, l) for l in range(L)]
    return {
        "x": x,
        "w_alpha": np.stack([d["w_alpha"] for d in wts]),
        "w_beta": np.stack([d["w_beta"] for d in wts]),
        "w_alpha_f32": np.stack([d["w_alpha_f32"] for d in wts]),
        "w_beta_f32": np.stack([d["w_beta_f32"] for d in wts]),
        "dt": np.stack([d["dt"] for d in lw]),
        "ssm_a": np.stack([d["ssm_a"] for d in lw]),
    }


# ---------------------------------------------------------------------------
# Weights of the two input projections (qkv: 10240 outputs, z: 6144 outputs)
# as dense BF16 ~ N(0, 1/sqrt(n_embd)), so that qkv and z come out about
# N(0, 1) like the decode workloads' qkv and z. The layer input x is ab_x.
# ---------------------------------------------------------------------------
def proj_head_weights(w: Workload, name: str, l: int, head: int, n_embd: int = N_EMBD) -> np.ndarray:
    """BF16 bit patterns [128][n_embd] of the rows of one 128-wide output head of layer l.

    ``name`` is "w_qkv" (80 heads: 16 q, 16 k, 48 v; rows 128 head .. 128 head + 127 of the
    10240) or "w_gate" (48 heads of z). Each (layer, head) block is its own Philox stream.
    """
    return to_bf16_bits(_normal(w.seed, name, (l, head), (HEAD_DIM, n_embd), std=1.0 / math.sqrt(n_embd)))


def proj_weights(w: Workload, l: int, n_embd: int = N_EMBD) -> dict:
    """BF16 bit patterns of layer l's w_qkv [10240][n_embd] and w_gate [6144][n_embd]."""
    return {
        "w_qkv": np.concatenate([proj_head_weights(w, "w_qkv", l, h, n_embd) for h in range(CONV_CHANNELS // HEAD_DIM)]),
        "w_gate": np.concatenate([proj_head_weights(w, "w_gate", l, h, n_embd) for h in range(VALUE_DIM // HEAD_DIM)]),
    }
