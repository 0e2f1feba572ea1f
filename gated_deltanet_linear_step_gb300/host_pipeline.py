"""Decode steps fed from host memory, with the copies overlapped with compute.

``HostDecodePipeline`` runs ``gdn_decode_step`` (or its varlen form) on
per-step activations that live in pinned host memory: each ``submit`` copies
one step's qkv, z, alpha and beta to the device, runs the step, and copies y
back. Two device slots alternate, and three CUDA streams carry the three
stages, so the host-to-device copy of step k + 1 and the device-to-host copy
of step k - 1 run while step k computes. Events order every reuse of a slot:

    copy-in k   waits for  step k - 2    (the slot's inputs are free)
    step k      waits for  copy-in k, and copy-out k - 2 (the slot's y is free)
    copy-out k  waits for  step k

The state and conv history stay on the device and are updated in place by the
steps in submission order. Each copy is one cudaMemcpyAsync issued by torch;
the step itself is the library's kernel through the C ABI.
"""
from __future__ import annotations

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
        self.dev = torch.device(device) if device is not None else state.device
        Bn, L, T = shape
        self.w = weights
        self.conv_state = conv_state
        self.state = state
        self.seq_len = seq_len
        widths = {"qkv": B.CONV_CHANNELS, "z": B.VALUE_DIM, "alpha": B.V_HEADS, "beta": B.V_HEADS}
        self.slots = [{k: torch.empty((Bn, L, T, widths[k]), device=self.dev) for k in self.IN_KEYS}
                      for _ in range(2)]
        for s in self.slots:
            s["y"] = torch.empty((Bn, L, T, B.VALUE_DIM), device=self.dev)
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_step = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_step = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.count = 0
        self.in_bytes = sum(t.numel() * t.element_size() for k, t in self.slots[0].items() if k != "y")
        self.out_bytes = self.slots[0]["y"].numel() * self.slots[0]["y"].element_size()

    def submit(self, host_in: dict, host_y: torch.Tensor) -> None:
        """Queues one step: ``host_in`` maps qkv, z, alpha, beta to pinned host tensors of
        the step's shapes; y is copied into the pinned ``host_y``. Returns at once; the
        host tensors must stay untouched until ``synchronize``."""
        k = self.count
        i = k % 2
        slot = self.slots[i]
        with torch.cuda.stream(self.s_in):
            if k >= 2:
                self.s_in.wait_event(self.ev_step[i])
            for key in self.IN_KEYS:
                slot[key].copy_(host_in[key], non_blocking=True)
            self.ev_in[i].record(self.s_in)
        self.s_step.wait_event(self.ev_in[i])
        if k >= 2:
            self.s_step.wait_event(self.ev_out[i])
        w = self.w
        if self.seq_len is None:
            B.gdn_decode_step(slot["qkv"], slot["z"], slot["alpha"], slot["beta"], w["dt"], w["ssm_a"], w["conv_w"],
                              w["ssm_norm"], self.conv_state, self.state, slot["y"], stream=self.s_step)
        else:
            B.gdn_decode_step_varlen(slot["qkv"], slot["z"], slot["alpha"], slot["beta"], w["dt"], w["ssm_a"],
                                     w["conv_w"], w["ssm_norm"], self.conv_state, self.state, slot["y"],
                                     self.seq_len, stream=self.s_step)
        self.ev_step[i].record(self.s_step)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_step[i])
            host_y.copy_(slot["y"], non_blocking=True)
            self.ev_out[i].record(self.s_out)
        self.count += 1

    def synchronize(self) -> None:
        """Waits for every submitted step and copy."""
        for s in (self.s_in, self.s_step, self.s_out):
            s.synchronize()
