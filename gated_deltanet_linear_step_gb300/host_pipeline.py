"""Decode steps fed from host memory, with the copies overlapped with compute.

``HostDecodePipeline`` wraps the library's native host pipeline
(``gdn_host_pipeline_*`` in ``include/gdn.h``): each ``submit`` queues the
host-to-device copies of one step's qkv, z, alpha and beta, the decode step,
and the copy of its y back to the host. Two device slots alternate and three
CUDA streams carry the three stages, ordered by events, so step k + 1's inputs
and step k - 1's y move while step k computes. This module only marshals
arguments; the slots are a device tensor it allocates and hands to the C ABI.
"""
from __future__ import annotations

import ctypes

import torch

from . import _binding as B


class HostDecodePipeline:
    """Double-buffered host-fed decode steps on one device.

    ``weights``: device tensors dt, ssm_a, conv_w, ssm_norm; ``conv_state`` and
    ``state``: device tensors updated in place; ``shape``: (B, L, T);
    ``seq_len``: optional device int32 [B] for ragged steps.
    """

    IN_KEYS = ("qkv", "z", "alpha", "beta")

    def __init__(self, weights: dict, conv_state: torch.Tensor, state: torch.Tensor, shape: tuple,
                 seq_len: torch.Tensor | None = None, device=None):
        lib = B.load_library()
        self.lib = lib
        self.dev = torch.device(device) if device is not None else state.device
        Bn, L, T = (int(v) for v in shape)
        self.shape = (Bn, L, T)
        dev = self.dev
        p = [
            B._ptr(weights["dt"], "dt", (L, B.V_HEADS), device=dev),
            B._ptr(weights["ssm_a"], "ssm_a", (L, B.V_HEADS), device=dev),
            B._ptr(weights["conv_w"], "conv_w", (L, B.CONV_CHANNELS, B.D_CONV), device=dev),
            B._ptr(weights["ssm_norm"], "ssm_norm", (L, B.HEAD_DIM), device=dev),
            B._ptr(conv_state, "conv_state", (Bn, L, B.CONV_CHANNELS, B.D_CONV - 1), device=dev),
            B._ptr(state, "state", (Bn, L, B.V_HEADS, B.HEAD_DIM, B.HEAD_DIM), device=dev),
            B._ptr(seq_len, "seq_len", (Bn,), dtype=torch.int32, device=dev, optional=True),
        ]
        n = int(lib.gdn_host_pipeline_slot_bytes(Bn, L, T))
        if n == 0:
            raise ValueError(f"sizes out of range: {shape}")
        self.slots = torch.empty(n, dtype=torch.uint8, device=dev)
        self.keep = (weights, conv_state, state, seq_len)  # the pipeline holds their pointers
        handle = ctypes.c_void_p()
        B._check(lib.gdn_host_pipeline_create(ctypes.byref(handle), *p, self.slots.data_ptr(), n, Bn, L, T,
                                              dev.index if dev.index is not None else torch.cuda.current_device()))
        self.handle = handle
        rows = Bn * L * T
        self.widths = {"qkv": B.CONV_CHANNELS, "z": B.VALUE_DIM, "alpha": B.V_HEADS, "beta": B.V_HEADS}
        self.in_bytes = sum(rows * w * 4 for w in self.widths.values())
        self.out_bytes = rows * B.VALUE_DIM * 4

    def _host(self, t, name, width):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or t.dtype != torch.float32:
            raise TypeError(f"{name} must be a float32 CPU tensor (pinned for overlapped copies)")
        if tuple(t.shape) != (*self.shape, width) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {(*self.shape, width)} tensor")
        return t.data_ptr()

    def submit(self, host_in: dict, host_y: torch.Tensor) -> None:
        """Queues one step: ``host_in`` maps qkv, z, alpha, beta to host tensors of the step's
        shapes; y is copied into ``host_y``. Returns at once; the host tensors must stay
        untouched until ``synchronize``."""
        ptrs = [self._host(host_in[k], k, self.widths[k]) for k in self.IN_KEYS]
        y = self._host(host_y, "y", B.VALUE_DIM)
        B._check(self.lib.gdn_host_pipeline_submit(self.handle, *ptrs, y))

    def synchronize(self) -> None:
        """Waits for every submitted step and copy."""
        B._check(self.lib.gdn_host_pipeline_synchronize(self.handle))

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.gdn_host_pipeline_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
