"""fp64 CPU oracle for the Gated DeltaNet (GDN) decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and its ``--impl reference`` arm) may import
or call anything here. The CUDA library and its Python binding never do, and
this module imports nothing from them: the two share no code. Only the seeded
input generators in ``workloads/`` serve both.

What it computes. The decode step of a GDN layer's recurrent mixer, in the
order spelled out by the header comment of the Winery-Strata page
``include/strata/core/layer.hpp`` (the operation-order list and its four
traps) and composed by ``gdn_layer`` on the page ``src/core/layer.cpp``
(steps 3 to 7). Per sequence b, layer l and valid token t:

1. causal depthwise conv of the 10240 qkv channels against the rolling
   conv_state (d_conv = 4, no bias), then the history shifts by one token;
2. SiLU on the whole 10240-wide conv output, before the q|k|v split;
3. L2 normalisation of each 128-wide q head and k head (16 each), eps 1e-6;
   v is not normalised;
4. q scaled by 1/sqrt(128) after its norm;
5. beta = sigmoid(beta_raw); g = softplus(alpha_raw + dt) * ssm_a;
   decay = exp(g);
6. the gated delta rule on each v head's 128x128 state, v head h reading
   q/k head h // 3:  S *= decay; kv = S^T k; d = (v - kv) * beta;
   S += k d^T; o = S^T q;
7. y = rms_norm(o per 128-wide head, ssm_norm, eps 1e-6) * sigmoid(z).

Tokens at or past a sequence's valid length (the verify window of the page
``src/core/verify.cpp``, its window and commit graphs) change nothing: the
state and conv_state are those after ``len`` tokens and y is left as NaN.

Readings taken where the pages are silent or ambiguous (each also listed with
its reason in the design notes):

* l2 norm form ``x / sqrt(sum x^2 + eps)``;
* RMSNorm form ``o / sqrt(mean o^2 + eps) * w`` over one 128-wide head, with
  one ssm_norm vector of 128 shared by all heads;
* softplus evaluated exactly as ``max(x, 0) + log1p(exp(-|x|))``;
* conv taps: ``w[c][0]`` multiplies the oldest history entry and ``w[c][3]``
  the current input; the history is stored oldest first as ``[C][3]``;
* state tile orientation ``S[i][j]``: i indexes k (rows), j indexes v
  (columns), so ``kv = S^T k`` reduces over rows;
* the input projections (``in_proj``) take dense BF16 weights and the float32
  layer input unrounded: the pages' qkv and gate weights are quantized packs
  that need trained values, and their BF16 path offers a float32-activation
  form.

Pinning. Every function here is pinned by ``tests/test_oracle_pins.py`` to
closed forms, exact rational arithmetic on tiny cases, invariants the
definition fixes, and the page's constants (``tests/golden/geometry.txt``).
The pages print no worked numeric example, so no function is pinned to a
printed value; none is left unpinned.

All arithmetic is float64 on the float32 inputs promoted exactly. The conv
state stays an exact copy of float32 inputs and is returned as float32.
"""
from __future__ import annotations

import math

import numpy as np

# Geometry (header comment of include/strata/core/layer.hpp and the q|k|v
# views in gdn_layer step 4 of src/core/layer.cpp).
HEAD_DIM = 128          # S, the state size of one head
K_HEADS = 16            # q heads = k heads
V_HEADS = 48            # v heads
CONV_CHANNELS = 10240   # q | k | v
VALUE_DIM = V_HEADS * HEAD_DIM
D_CONV = 4
Q_OFFSET = 0
K_OFFSET = K_HEADS * HEAD_DIM           # 2048
V_OFFSET = 2 * K_HEADS * HEAD_DIM       # 4096
EPS = 1e-6              # the layer's RMS epsilon, used for both norms


# ---------------------------------------------------------------- step 1 --
def causal_conv(x: np.ndarray, conv_state: np.ndarray, conv_w: np.ndarray) -> np.ndarray:
    """Depthwise causal conv output for one token.

    ``xc[c] = sum_{j<3} w[c][j] * hist[c][j] + w[c][3] * x[c]`` with
    ``hist[c][0]`` the oldest input. No bias: the layer loads only the conv
    weight (src/core/layer.cpp, gdn_layer's weight list).
    """
    x = np.asarray(x, np.float64)
    hist = np.asarray(conv_state, np.float64)
    w = np.asarray(conv_w, np.float64)
    xc = np.zeros_like(x)
    for j in range(D_CONV - 1):
        xc += w[:, j] * hist[:, j]
    xc += w[:, D_CONV - 1] * x
    return xc


def roll_conv_state(conv_state: np.ndarray, x: np.ndarray) -> np.ndarray:
    """The history after one token: drop the oldest entry, append x (an exact copy)."""
    hist = np.asarray(conv_state, np.float32)
    out = np.empty_like(hist)
    out[:, : D_CONV - 2] = hist[:, 1:]
    out[:, D_CONV - 2] = np.asarray(x, np.float32)
    return out


# ---------------------------------------------------------------- step 2 --
def sigmoid(x):
    x = np.asarray(x, np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """x * sigmoid(x)."""
    x = np.asarray(x, np.float64)
    return x * sigmoid(x)


def softplus(x):
    """log(1 + exp(x)), evaluated as max(x, 0) + log1p(exp(-|x|)) so it never overflows."""
    x = np.asarray(x, np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


# ---------------------------------------------------------------- step 3 --
def l2_normalize(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """x / sqrt(sum(x^2) + eps) over the last axis (one 128-wide head per row)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------- step 5 --
def gates(alpha_raw, beta_raw, dt, ssm_a):
    """Per-v-head gates: beta = sigmoid(beta_raw), decay = exp(softplus(alpha_raw + dt) * ssm_a)."""
    beta = sigmoid(beta_raw)
    g = softplus(np.asarray(alpha_raw, np.float64) + np.asarray(dt, np.float64)) * np.asarray(ssm_a, np.float64)
    return beta, np.exp(g)


def ab_gates(x, w_alpha, w_beta, dt, ssm_a):
    """The alpha/beta projections with their gate epilogue (the fused_gdn_ab stage of
    gdn_layer step 5 on src/core/layer.cpp): alpha_raw = x . w_alpha[h], beta_raw =
    x . w_beta[h]; returns (gate, beta) with gate = softplus(alpha_raw + dt) * ssm_a,
    the log of the decay, and beta = sigmoid(beta_raw).

    ``x`` is [..., n_embd]; the weights are [48][n_embd] (the BF16 values, exactly as
    float); ``dt`` and ``ssm_a`` are [48].
    """
    x = np.asarray(x, np.float64)
    alpha_raw = x @ np.asarray(w_alpha, np.float64).T
    beta_raw = x @ np.asarray(w_beta, np.float64).T
    gate = softplus(alpha_raw + np.asarray(dt, np.float64)) * np.asarray(ssm_a, np.float64)
    return gate, sigmoid(beta_raw)



def in_proj(x, w_qkv, w_gate):
    """The mixer's two input projections of the layer input: qkv = w_qkv x, the
    10240 conv channels q|k|v (gdn_layer step 2 on src/core/layer.cpp), and
    z = w_gate x, the 6144-wide output gate (the start of gdn_layer step 7).

    The weights are dense BF16 matrices [n_out][n_embd], passed as their exact
    float values; ``x`` is [..., n_embd]. Returns (qkv, z) in float64, with no
    rounding of x or of the products.
    """
    x = np.asarray(x, np.float64)
    qkv = x @ np.asarray(w_qkv, np.float64).T
    z = x @ np.asarray(w_gate, np.float64).T
    return qkv, z

# ---------------------------------------------------------------- step 6 --
def delta_rule_step(S, k, q, v, beta, decay):
    """One gated delta-rule step on one head's state, in the definition's order.

    ``S`` is (dk, dv): rows follow k and q, columns follow v. Returns the new
    state and the readout ``o = S_new^T q``.
    """
    S = np.asarray(S, np.float64) * decay          # S *= decay
    k = np.asarray(k, np.float64)
    q = np.asarray(q, np.float64)
    kv = S.T @ k                                   # kv = S^T k
    d = (np.asarray(v, np.float64) - kv) * beta    # d = (v - kv) * beta
    S = S + np.outer(k, d)                         # S += k d^T
    o = S.T @ q                                    # o = S^T q
    return S, o


# ---------------------------------------------------------------- step 7 --
def gated_rms_norm(o, z, w, eps: float = EPS, gate: str = "sigmoid"):
    """rms_norm(o over its last axis) * w * gate(z); the gate is sigmoid (or SiLU, the earlier variant)."""
    o = np.asarray(o, np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    gz = sigmoid(z) if gate == "sigmoid" else silu(z)
    return o / rms * np.asarray(w, np.float64) * gz


# ------------------------------------------------------------ steps 1-5 --
def preprocess_token(x, conv_state, conv_w, alpha_raw, beta_raw, dt, ssm_a, gates_ready: bool = False):
    """Steps 1-5 for one token of one (sequence, layer). With ``gates_ready``,
    ``alpha_raw`` already holds the log decay and ``beta_raw`` holds beta (the
    outputs of ``ab_gates``).

    Returns a dict with the normalised and scaled q (16x128), the normalised
    k (16x128), v (48x128), beta and decay (48 each), the conv output before
    SiLU (``xc``) and the new conv history (float32).
    """
    xc = causal_conv(x, conv_state, conv_w)
    h = silu(xc)                                          # whole 10240 channels
    q = h[Q_OFFSET:K_OFFSET].reshape(K_HEADS, HEAD_DIM)
    k = h[K_OFFSET:V_OFFSET].reshape(K_HEADS, HEAD_DIM)
    v = h[V_OFFSET:].reshape(V_HEADS, HEAD_DIM)           # not normalised
    q = l2_normalize(q) * (1.0 / math.sqrt(HEAD_DIM))     # scale after the norm
    k = l2_normalize(k)
    if gates_ready:
        beta, decay = np.asarray(beta_raw, np.float64), np.exp(np.asarray(alpha_raw, np.float64))
    else:
        beta, decay = gates(alpha_raw, beta_raw, dt, ssm_a)
    return {"q": q, "k": k, "v": v, "beta": beta, "decay": decay, "xc": xc,
            "conv_state": roll_conv_state(conv_state, x)}


def v_head_to_k_head(h: int) -> int:
    """v head h reads q/k head h // 3 (48 v heads over 16 k heads)."""
    return h // (V_HEADS // K_HEADS)


def gdn_layer_step(x, z, alpha_raw, beta_raw, dt, ssm_a, conv_w, ssm_norm, conv_state, state,
                   gate: str = "sigmoid", gates_ready: bool = False):
    """Steps 1-7 for one token of one (sequence, layer).

    ``state`` is (48, 128, 128). Returns (y (6144,), new state, new conv history).
    """
    p = preprocess_token(x, conv_state, conv_w, alpha_raw, beta_raw, dt, ssm_a, gates_ready)
    new_state = np.empty((V_HEADS, HEAD_DIM, HEAD_DIM), np.float64)
    o = np.empty((V_HEADS, HEAD_DIM), np.float64)
    for h in range(V_HEADS):
        kh = v_head_to_k_head(h)
        new_state[h], o[h] = delta_rule_step(state[h], p["k"][kh], p["q"][kh], p["v"][h],
                                             p["beta"][h], p["decay"][h])
    zz = np.asarray(z, np.float64).reshape(V_HEADS, HEAD_DIM)
    y = gated_rms_norm(o, zz, ssm_norm, gate=gate).reshape(VALUE_DIM)
    return y, new_state, p["conv_state"]


def gdn_decode(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state,
               seq_len=None, gate: str = "sigmoid", gates_ready: bool = False):
    """The whole decode call: B sequences x L layers x T tokens.

    Shapes (outermost first): qkv [B][L][T][10240], z [B][L][T][6144],
    alpha/beta [B][L][T][48], dt/ssm_a [L][48], conv_w [L][10240][4],
    ssm_norm [L][128], conv_state [B][L][10240][3], state
    [B][L][48][128][128]; ``seq_len`` [B] (valid tokens per sequence) or None
    for all T.

    Returns ``(y, state_out, conv_state_out)``: y float64 [B][L][T][6144] with
    NaN for tokens at or past seq_len; state_out float64; conv_state_out
    float32 (an exact copy of inputs).
    """
    qkv = np.asarray(qkv)
    B, L, T = qkv.shape[:3]
    y = np.empty((B, L, T, VALUE_DIM), np.float64)
    state_out = np.empty((B, L, V_HEADS, HEAD_DIM, HEAD_DIM), np.float64)
    conv_out = np.empty((B, L, CONV_CHANNELS, D_CONV - 1), np.float32)
    for b in range(B):
        n = T if seq_len is None else int(seq_len[b])
        for l in range(L):
            sl = {"qkv": qkv[b, l], "z": z[b, l], "alpha": alpha[b, l], "beta": beta[b, l],
                  "conv_state": conv_state[b, l], "state": state[b, l]}
            wts = {"dt": dt[l], "ssm_a": ssm_a[l], "conv_w": conv_w[l], "ssm_norm": ssm_norm[l]}
            y[b, l], state_out[b, l], conv_out[b, l] = gdn_decode_slice(sl, wts, n, gate=gate,
                                                                        gates_ready=gates_ready)
    return y, state_out, conv_out


def gdn_decode_slice(sl: dict, wts: dict, n: int | None = None, gate: str = "sigmoid", gates_ready: bool = False):
    """``gdn_decode`` for one (sequence, layer): ``sl`` holds qkv [T][C], z, alpha,
    beta, conv_state, state; ``wts`` holds dt, ssm_a, conv_w, ssm_norm of the layer.

    Returns (y [T][6144] with NaN past n, state [48][128][128] float64, conv_state float32).
    """
    T = sl["qkv"].shape[0]
    n = T if n is None else n
    y = np.full((T, VALUE_DIM), np.nan)
    st = np.asarray(sl["state"], np.float64)
    cs = np.asarray(sl["conv_state"], np.float32)
    for t in range(n):
        y[t], st, cs = gdn_layer_step(sl["qkv"][t], sl["z"][t], sl["alpha"][t], sl["beta"][t], wts["dt"],
                                      wts["ssm_a"], wts["conv_w"], wts["ssm_norm"], cs, st, gate=gate,
                                      gates_ready=gates_ready)
    return y, st, cs
