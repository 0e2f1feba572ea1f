"""Thin ctypes binding of ``libgdn.so`` (C ABI in ``include/gdn.h``).

Argument marshalling only: every step of the decode path runs in the CUDA
kernel behind the C ABI. Functions take contiguous CUDA torch tensors, derive
B, L and T from ``qkv``'s shape, check every other tensor's shape, and pass
raw device pointers plus the stream (the current torch stream of the
tensors' device unless one is given). A non-OK status raises ``GdnError``
with the library's message. There is no fallback: without the built library
every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

HEAD_DIM = 128
K_HEADS = 16
V_HEADS = 48
CONV_CHANNELS = 10240
VALUE_DIM = 6144
D_CONV = 4

FLAG_NO_STATE_WRITE = 0x1
FLAG_NO_Y = 0x2
FLAG_SILU_GATE = 0x4
FLAG_GATES_READY = 0x8
FLAG_TEST_GIVE_UP = 0x10  # tests only: the first wait for a state tile gives up (see gdn.h)

STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_ALIGN", 4: "GDN_ERR_ALIAS",
          5: "GDN_ERR_CUDA", 6: "GDN_ERR_FLAGS"}


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads ``libgdn.so`` once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        step_args = [_P] * 11 + [_I, _I, _I, _P]
        lib.gdn_decode_step.argtypes = step_args
        lib.gdn_decode_step_varlen.argtypes = [_P] * 12 + [_I, _I, _I, _P]
        lib.gdn_verify_window.argtypes = [_P] * 12 + [_I, _I, _I, _P]
        lib.gdn_verify_commit.argtypes = [_P] * 9 + [_I, _I, _I, _P]
        lib.gdn_decode_step_ex.argtypes = [_P] * 12 + [_I, _I, _I, ctypes.c_uint32, _P]
        lib.gdn_ab_gates.argtypes = [_P] * 7 + [_I, _I, _I, _I, _P]
        lib.gdn_in_proj.argtypes = [_P] * 6 + [ctypes.c_size_t, _I, _I, _I, _I, _P]
        lib.gdn_in_proj_noalloc.argtypes = [_P] * 5 + [_I, _I, _I, _I, _P]
        lib.gdn_step_inputs.argtypes = [_P] * 12 + [ctypes.c_size_t, _I, _I, _I, _I, _P]
        lib.gdn_in_proj_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.gdn_proj_pack_bytes.argtypes = [_I, _I]
        lib.gdn_proj_pack_bytes.restype = ctypes.c_size_t
        lib.gdn_pack_proj_weights.argtypes = [_P] * 5 + [ctypes.c_size_t, _I, _I, _P]
        lib.gdn_in_proj_packed.argtypes = [_P, _P, ctypes.c_size_t, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _P]
        lib.gdn_step_inputs_packed.argtypes = [_P, _P, ctypes.c_size_t] + [_P] * 7 + [ctypes.c_size_t, _I, _I, _I,
                                                                                        _I, _P]
        lib.gdn_host_pipeline_slot_bytes.argtypes = [_I, _I, _I]
        lib.gdn_host_pipeline_slot_bytes.restype = ctypes.c_size_t
        lib.gdn_host_pipeline_create.argtypes = [ctypes.POINTER(ctypes.c_void_p)] + [_P] * 8 + [ctypes.c_size_t, _I,
                                                                                               _I, _I, _I]
        lib.gdn_host_pipeline_submit.argtypes = [_P] * 6
        lib.gdn_host_pipeline_synchronize.argtypes = [_P]
        lib.gdn_host_pipeline_destroy.argtypes = [_P]
        lib.gdn_host_pipeline_destroy.restype = None
        lib.gdn_in_proj_workspace_size.restype = ctypes.c_size_t
        for fn in ("gdn_decode_step", "gdn_decode_step_varlen", "gdn_verify_window", "gdn_verify_commit",
                   "gdn_decode_step_ex", "gdn_ab_gates", "gdn_in_proj", "gdn_in_proj_noalloc", "gdn_step_inputs",
                   "gdn_pack_proj_weights", "gdn_in_proj_packed", "gdn_step_inputs_packed", "gdn_host_pipeline_create",
                   "gdn_host_pipeline_submit", "gdn_host_pipeline_synchronize", "gdn_get_geometry",
                   "gdn_read_device_error"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.gdn_get_geometry.argtypes = [ctypes.POINTER(ctypes.c_int32)]
        lib.gdn_read_device_error.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_dispatch_kernel.argtypes = [_I, _I, _I]
        lib.gdn_dispatch_kernel.restype = ctypes.c_int
        _lib = lib
    return _lib


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode()


def _check(status: int):
    if status != 0:
        raise GdnError(status, gdn_last_error())


def _ptr(t, name, shape, dtype=torch.float32, device=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _shapes(qkv):
    if not isinstance(qkv, torch.Tensor) or qkv.dim() != 4 or qkv.shape[3] != CONV_CHANNELS:
        raise ValueError(f"qkv must be a [B][L][T][{CONV_CHANNELS}] tensor")
    B, L, T = (int(s) for s in qkv.shape[:3])
    return B, L, T


def _step_ptrs(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, need_y=True):
    B, L, T = _shapes(qkv)
    dev = qkv.device
    return (B, L, T, dev, [
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev, optional=not need_y),
        _ptr(alpha, "alpha", (B, L, T, V_HEADS), device=dev),
        _ptr(beta, "beta", (B, L, T, V_HEADS), device=dev),
        _ptr(dt, "dt", (L, V_HEADS), device=dev),
        _ptr(ssm_a, "ssm_a", (L, V_HEADS), device=dev),
        _ptr(conv_w, "conv_w", (L, CONV_CHANNELS, D_CONV), device=dev),
        _ptr(ssm_norm, "ssm_norm", (L, HEAD_DIM), device=dev, optional=not need_y),
        _ptr(conv_state, "conv_state", (B, L, CONV_CHANNELS, D_CONV - 1), device=dev),
        _ptr(state, "state", (B, L, V_HEADS, HEAD_DIM, HEAD_DIM), device=dev),
        _ptr(y, "y", (B, L, T, VALUE_DIM), device=dev, optional=not need_y),
    ])


def gdn_decode_step(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, stream=None):
    """One decode call over T tokens; updates ``conv_state`` and ``state`` in place and writes ``y``."""
    lib = load_library()
    B, L, T, dev, p = _step_ptrs(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y)
    with torch.cuda.device(dev):
        _check(lib.gdn_decode_step(*p, B, L, T, _stream_handle(stream, dev)))


def gdn_decode_step_varlen(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, seq_len,
                           stream=None):
    """``gdn_decode_step`` applying only the first ``seq_len[b]`` tokens of sequence b (int32 [B] on the device)."""
    lib = load_library()
    B, L, T, dev, p = _step_ptrs(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y)
    sl = _ptr(seq_len, "seq_len", (B,), dtype=torch.int32, device=dev, optional=True)
    with torch.cuda.device(dev):
        _check(lib.gdn_decode_step_varlen(*p, sl, B, L, T, _stream_handle(stream, dev)))


def gdn_verify_window(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, seq_len=None,
                      stream=None):
    """Phase 1 of a verify window: y for the draft tokens; ``state`` and ``conv_state`` are only read."""
    lib = load_library()
    B, L, T, dev, p = _step_ptrs(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y)
    sl = _ptr(seq_len, "seq_len", (B,), dtype=torch.int32, device=dev, optional=True)
    with torch.cuda.device(dev):
        _check(lib.gdn_verify_window(*p, sl, B, L, T, _stream_handle(stream, dev)))


def gdn_verify_commit(qkv, alpha, beta, dt, ssm_a, conv_w, conv_state, state, n_keep, stream=None):
    """Phase 2: advance ``state`` and ``conv_state`` by ``n_keep[b]`` accepted tokens (int32 [B] on the device)."""
    lib = load_library()
    B, L, T = _shapes(qkv)
    dev = qkv.device
    p = [
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(alpha, "alpha", (B, L, T, V_HEADS), device=dev),
        _ptr(beta, "beta", (B, L, T, V_HEADS), device=dev),
        _ptr(dt, "dt", (L, V_HEADS), device=dev),
        _ptr(ssm_a, "ssm_a", (L, V_HEADS), device=dev),
        _ptr(conv_w, "conv_w", (L, CONV_CHANNELS, D_CONV), device=dev),
        _ptr(conv_state, "conv_state", (B, L, CONV_CHANNELS, D_CONV - 1), device=dev),
        _ptr(state, "state", (B, L, V_HEADS, HEAD_DIM, HEAD_DIM), device=dev),
        _ptr(n_keep, "n_keep", (B,), dtype=torch.int32, device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_verify_commit(*p, B, L, T, _stream_handle(stream, dev)))


def gdn_decode_step_ex(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, seq_len=None,
                       flags=0, stream=None):
    """``gdn_decode_step_varlen`` with ``FLAG_*`` bits (no state write, no y, SiLU output gate)."""
    lib = load_library()
    need_y = not (flags & FLAG_NO_Y)
    B, L, T, dev, p = _step_ptrs(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y,
                                 need_y=need_y)
    sl = _ptr(seq_len, "seq_len", (B,), dtype=torch.int32, device=dev, optional=True)
    with torch.cuda.device(dev):
        _check(lib.gdn_decode_step_ex(*p, sl, B, L, T, int(flags), _stream_handle(stream, dev)))


def gdn_ab_gates(x, w_alpha, w_beta, dt, ssm_a, gate, beta, stream=None):
    """alpha/beta projections with the gate epilogue: writes the log decay to ``gate`` and
    sigmoid(beta_raw) to ``beta`` ([B][L][T][48]); the weights are [L][48][n_embd] BF16
    (torch.bfloat16, or their bit patterns as int16/uint16)."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    for name, w in (("w_alpha", w_alpha), ("w_beta", w_beta)):
        _bf16_weight(w, name)
    p = [
        _ptr(x, "x", (B, L, T, E), device=dev),
        _ptr(w_alpha, "w_alpha", (L, V_HEADS, E), dtype=w_alpha.dtype, device=dev),
        _ptr(w_beta, "w_beta", (L, V_HEADS, E), dtype=w_beta.dtype, device=dev),
        _ptr(dt, "dt", (L, V_HEADS), device=dev),
        _ptr(ssm_a, "ssm_a", (L, V_HEADS), device=dev),
        _ptr(gate, "gate", (B, L, T, V_HEADS), device=dev),
        _ptr(beta, "beta", (B, L, T, V_HEADS), device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_ab_gates(*p, B, L, T, E, _stream_handle(stream, dev)))


def _bf16_weight(w, name):
    if not isinstance(w, torch.Tensor) or w.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must hold BF16 values (torch.bfloat16) or their 16-bit patterns")
    return w


def gdn_in_proj_workspace_size(B: int, L: int, T: int, n_embd: int) -> int:
    """Bytes of device workspace gdn_in_proj needs (0 for sizes out of range)."""
    return int(load_library().gdn_in_proj_workspace_size(int(B), int(L), int(T), int(n_embd)))


def gdn_in_proj(x, w_qkv, w_gate, qkv, z, workspace, stream=None):
    """The qkv and z input projections on the tensor cores: qkv = w_qkv x ([B][L][T][10240])
    and z = w_gate x ([B][L][T][6144]). The weights are [L][10240][n_embd] and
    [L][6144][n_embd] BF16 (torch.bfloat16, or their bit patterns as int16/uint16);
    ``workspace`` is a uint8 CUDA tensor of at least gdn_in_proj_workspace_size() bytes."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    for name, w in (("w_qkv", w_qkv), ("w_gate", w_gate)):
        _bf16_weight(w, name)
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 or workspace.dim() != 1:
        raise TypeError("workspace must be a 1-D torch.uint8 tensor")
    p = [
        _ptr(x, "x", (B, L, T, E), device=dev),
        _ptr(w_qkv, "w_qkv", (L, CONV_CHANNELS, E), dtype=w_qkv.dtype, device=dev),
        _ptr(w_gate, "w_gate", (L, VALUE_DIM, E), dtype=w_gate.dtype, device=dev),
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev),
        _ptr(workspace, "workspace", tuple(workspace.shape), dtype=torch.uint8, device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_in_proj(*p, int(workspace.numel()), B, L, T, E, _stream_handle(stream, dev)))


def gdn_step_inputs(x, w_qkv, w_gate, w_alpha, w_beta, dt, ssm_a, qkv, z, gate, beta, workspace, stream=None):
    """All four decode-step inputs from the layer input on the tensor cores: qkv and z as
    gdn_in_proj, gate (log decay) and beta as gdn_ab_gates. Weights are BF16 (torch.bfloat16,
    or their 16-bit patterns); ``workspace`` as for gdn_in_proj."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    for name, w in (("w_qkv", w_qkv), ("w_gate", w_gate), ("w_alpha", w_alpha), ("w_beta", w_beta)):
        _bf16_weight(w, name)
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 or workspace.dim() != 1:
        raise TypeError("workspace must be a 1-D torch.uint8 tensor")
    p = [
        _ptr(x, "x", (B, L, T, E), device=dev),
        _ptr(w_qkv, "w_qkv", (L, CONV_CHANNELS, E), dtype=w_qkv.dtype, device=dev),
        _ptr(w_gate, "w_gate", (L, VALUE_DIM, E), dtype=w_gate.dtype, device=dev),
        _ptr(w_alpha, "w_alpha", (L, V_HEADS, E), dtype=w_alpha.dtype, device=dev),
        _ptr(w_beta, "w_beta", (L, V_HEADS, E), dtype=w_beta.dtype, device=dev),
        _ptr(dt, "dt", (L, V_HEADS), device=dev),
        _ptr(ssm_a, "ssm_a", (L, V_HEADS), device=dev),
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev),
        _ptr(gate, "gate", (B, L, T, V_HEADS), device=dev),
        _ptr(beta, "beta", (B, L, T, V_HEADS), device=dev),
        _ptr(workspace, "workspace", tuple(workspace.shape), dtype=torch.uint8, device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_step_inputs(*p, int(workspace.numel()), B, L, T, E, _stream_handle(stream, dev)))


def gdn_in_proj_noalloc(x, w_qkv, w_gate, qkv, z, stream=None):
    """gdn_in_proj with the split of x in the library's fixed 48 MiB scratch array instead of
    a caller workspace; calls on one device must not overlap in time."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    for name, w in (("w_qkv", w_qkv), ("w_gate", w_gate)):
        _bf16_weight(w, name)
    p = [
        _ptr(x, "x", (B, L, T, E), device=dev),
        _ptr(w_qkv, "w_qkv", (L, CONV_CHANNELS, E), dtype=w_qkv.dtype, device=dev),
        _ptr(w_gate, "w_gate", (L, VALUE_DIM, E), dtype=w_gate.dtype, device=dev),
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_in_proj_noalloc(*p, B, L, T, E, _stream_handle(stream, dev)))


def gdn_proj_pack_bytes(L: int, n_embd: int) -> int:
    """Bytes of the packed projection weights of L layers (0 for sizes out of range)."""
    return int(load_library().gdn_proj_pack_bytes(int(L), int(n_embd)))


def _packed(packed, dev):
    if not isinstance(packed, torch.Tensor) or packed.dtype != torch.uint8 or packed.dim() != 1:
        raise TypeError("packed must be a 1-D torch.uint8 tensor written by gdn_pack_proj_weights")
    return _ptr(packed, "packed", tuple(packed.shape), dtype=torch.uint8, device=dev), int(packed.numel())


def gdn_pack_proj_weights(w_qkv, w_gate, packed, w_alpha=None, w_beta=None, stream=None):
    """Rearranges the projection weights into ``packed`` (a 1-D uint8 CUDA tensor of at least
    gdn_proj_pack_bytes(L, n_embd) bytes), the order gdn_in_proj_packed and
    gdn_step_inputs_packed read. w_alpha and w_beta are optional (zero rows without them)."""
    lib = load_library()
    _bf16_weight(w_qkv, "w_qkv")
    if w_qkv.dim() != 3:
        raise ValueError("w_qkv must be [L][10240][n_embd]")
    L, E = int(w_qkv.shape[0]), int(w_qkv.shape[2])
    dev = w_qkv.device
    if (w_alpha is None) != (w_beta is None):
        raise ValueError("give both w_alpha and w_beta, or neither")
    p = [
        _ptr(w_qkv, "w_qkv", (L, CONV_CHANNELS, E), dtype=w_qkv.dtype, device=dev),
        _ptr(_bf16_weight(w_gate, "w_gate"), "w_gate", (L, VALUE_DIM, E), dtype=w_gate.dtype, device=dev),
        None if w_alpha is None else _ptr(_bf16_weight(w_alpha, "w_alpha"), "w_alpha", (L, V_HEADS, E),
                                          dtype=w_alpha.dtype, device=dev),
        None if w_beta is None else _ptr(_bf16_weight(w_beta, "w_beta"), "w_beta", (L, V_HEADS, E),
                                         dtype=w_beta.dtype, device=dev),
    ]
    pp, nbytes = _packed(packed, dev)
    with torch.cuda.device(dev):
        _check(lib.gdn_pack_proj_weights(*p, pp, nbytes, L, E, _stream_handle(stream, dev)))


def gdn_in_proj_packed(x, packed, qkv, z, workspace, stream=None):
    """gdn_in_proj on weights packed by gdn_pack_proj_weights; bit-identical outputs."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 or workspace.dim() != 1:
        raise TypeError("workspace must be a 1-D torch.uint8 tensor")
    pp, nbytes = _packed(packed, dev)
    p = [
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev),
        _ptr(workspace, "workspace", tuple(workspace.shape), dtype=torch.uint8, device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_in_proj_packed(_ptr(x, "x", (B, L, T, E), device=dev), pp, nbytes, *p,
                                      int(workspace.numel()), B, L, T, E, _stream_handle(stream, dev)))


def gdn_step_inputs_packed(x, packed, dt, ssm_a, qkv, z, gate, beta, workspace, stream=None):
    """gdn_step_inputs on weights packed by gdn_pack_proj_weights (with w_alpha and w_beta);
    bit-identical outputs."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [B][L][T][n_embd] tensor")
    B, L, T, E = (int(v) for v in x.shape)
    dev = x.device
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 or workspace.dim() != 1:
        raise TypeError("workspace must be a 1-D torch.uint8 tensor")
    pp, nbytes = _packed(packed, dev)
    p = [
        _ptr(dt, "dt", (L, V_HEADS), device=dev),
        _ptr(ssm_a, "ssm_a", (L, V_HEADS), device=dev),
        _ptr(qkv, "qkv", (B, L, T, CONV_CHANNELS), device=dev),
        _ptr(z, "z", (B, L, T, VALUE_DIM), device=dev),
        _ptr(gate, "gate", (B, L, T, V_HEADS), device=dev),
        _ptr(beta, "beta", (B, L, T, V_HEADS), device=dev),
        _ptr(workspace, "workspace", tuple(workspace.shape), dtype=torch.uint8, device=dev),
    ]
    with torch.cuda.device(dev):
        _check(lib.gdn_step_inputs_packed(_ptr(x, "x", (B, L, T, E), device=dev), pp, nbytes, *p,
                                          int(workspace.numel()), B, L, T, E, _stream_handle(stream, dev)))


DISPATCH_KERNELS = {1: "gdn_decode_t1_kernel", 2: "gdn_window_kernel", 3: "gdn_chunk_kernel", 4: "gdn_window_tc_kernel"}


def gdn_dispatch_kernel(B: int, L: int, T: int, device=None) -> str:
    """Name of the kernel a decode call of B x L x T runs on the device (launches nothing)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        k = load_library().gdn_dispatch_kernel(int(B), int(L), int(T))
    if k < 0:
        raise GdnError(5 if B >= 1 and L >= 1 and 1 <= T else 2, gdn_last_error())
    return DISPATCH_KERNELS[k]


def gdn_get_geometry() -> dict:
    out = (ctypes.c_int32 * 8)()
    _check(load_library().gdn_get_geometry(out))
    keys = ("head_dim", "k_heads", "v_heads", "conv_channels", "value_dim", "d_conv", "max_t", "cta_threads")
    return dict(zip(keys, list(out)))


def gdn_read_device_error(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the kernel's device error word."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    out = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        _check(load_library().gdn_read_device_error(_stream_handle(stream, dev), ctypes.byref(out)))
    return int(out.value)
