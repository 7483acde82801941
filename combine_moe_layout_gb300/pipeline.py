"""One dispatch/combine step through the C ABI, with torch for device memory.

``MoeStep`` owns the device buffers of one problem size and runs
layout -> dispatch -> experts -> combine on a stream. The experts are the
synthetic ones of the workloads: identity for bf16 steps (combine reads the
receive buffer itself) and ``moe_expert_stub`` for fp8 steps.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _binding as B


@dataclass
class DeviceInputs:
    topk_idx: torch.Tensor      # [R][T][k] int32
    topk_weights: torch.Tensor  # [R][T][k] float32
    x: torch.Tensor             # [R][T][H] uint8 (fp8 codes) or bfloat16
    x_scales: torch.Tensor | None


def to_pinned_host(inputs) -> DeviceInputs:
    """The generated inputs in pinned host memory, for kernels that read them
    directly over the CPU-GPU link (bf16 bits are reinterpreted, not converted)."""
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    x = t(inputs.x)
    if x.dtype == torch.uint16:
        x = x.view(torch.bfloat16)
    return DeviceInputs(t(inputs.topk_idx), t(inputs.topk_weights), x,
                        None if inputs.x_scales is None else t(inputs.x_scales))


def to_device(inputs, device, pin: bool = False) -> DeviceInputs:
    """Copy generated numpy inputs to the device (bf16 bits are reinterpreted, not converted)."""
    def t(a):
        ht = torch.from_numpy(np.ascontiguousarray(a))
        if pin:
            ht = ht.pin_memory()
        return ht.to(device, non_blocking=pin)

    x = t(inputs.x)
    if x.dtype == torch.uint16:
        x = x.view(torch.bfloat16)
    elif x.dtype != torch.uint8:
        raise ValueError("x must hold uint16 bf16 bits or uint8 e4m3 codes")
    return DeviceInputs(t(inputs.topk_idx), t(inputs.topk_weights), x,
                        None if inputs.x_scales is None else t(inputs.x_scales))


class MoeStep:
    def __init__(self, workload, device="cuda", num_sms: int = 0, buffers: B.MoeBuffers | None = None):
        self.w = workload
        self.desc = B.MoeDesc.of(workload, num_sms)
        self.fp8 = workload.dtype != "bf16"  # slots hold e4m3 rows + scales
        self.device = torch.device(device)
        self.buf = buffers if buffers is not None else B.allocate_buffers(self.desc, self.device)
        self.slots = workload.num_experts * workload.num_ranks * workload.max_m
        if self.buf.expert_out is not None:
            self.y = self.buf.expert_out
        else:  # identity experts: combine reads the dispatched rows themselves
            self.y = self.buf.recv_x.view(torch.bfloat16).view(self.slots, workload.hidden)

    def reset(self, stream=None):
        B.moe_reset(self.desc, self.buf.flags, self.buf.err, stream)

    def layout(self, d: DeviceInputs, stream=None):
        b = self.buf
        B.moe_layout(self.desc, d.topk_idx, b.counts, b.flags, b.tok_slot, b.err, stream)

    def dispatch(self, d: DeviceInputs, stream=None):
        b = self.buf
        B.moe_dispatch(self.desc, d.x, d.x_scales, b.tok_slot, b.flags, b.recv_x, b.recv_scales, b.recv_meta, b.err,
                       stream)

    def layout_dispatch(self, d: DeviceInputs, stream=None):
        b = self.buf
        B.moe_layout_dispatch(self.desc, d.topk_idx, d.x, d.x_scales, b.counts, b.flags, b.tok_slot, b.recv_x,
                              b.recv_scales, b.recv_meta, b.err, stream)

    def experts(self, stream=None):
        if self.fp8:
            b = self.buf
            B.moe_expert_stub(self.desc, b.recv_x, b.recv_scales, b.counts, b.expert_out, b.err, stream)

    def combine(self, d: DeviceInputs, stream=None, out=None):
        """out: the step's output buffer (default: the device buffer; may be pinned host memory)."""
        b = self.buf
        B.moe_combine(self.desc, self.y, d.topk_weights, b.tok_slot, b.flags, b.out if out is None else out, b.err,
                      stream)

    def run(self, d: DeviceInputs, stream=None, fused: bool = False):
        if fused:
            self.layout_dispatch(d, stream)
        else:
            self.layout(d, stream)
            self.dispatch(d, stream)
        self.experts(stream)
        self.combine(d, stream)

    def recv(self, packed: B.PackedBuffers, stream=None):
        """The receive hook: wait for the counts, pack the filled slots expert-major."""
        b = self.buf
        B.moe_dispatch_recv(self.desc, b.counts, b.flags, b.recv_x, b.recv_scales, b.recv_meta, b.tok_slot,
                            packed.region_offsets, packed.packed_x, packed.packed_scales, packed.packed_meta,
                            packed.tok_packed, b.err, stream)

    def combine_packed(self, d: DeviceInputs, packed_y: torch.Tensor, packed: B.PackedBuffers, stream=None,
                       out=None):
        b = self.buf
        B.moe_combine_packed(self.desc, packed_y, packed.tok_packed, d.topk_weights, b.flags,
                             b.out if out is None else out, b.err, stream)

    def expert_mlp(self, weights, packed: B.PackedBuffers, h: torch.Tensor, packed_y: torch.Tensor, stream=None):
        """The expert stage on the packed rows: linear 1 with SwiGLU into h [R*T*k][I],
        then linear 2 into packed_y [R*T*k][H] (what combine_packed reads)."""
        b = self.buf
        B.moe_expert_gate_up(self.desc, weights.inter, packed.region_offsets, packed.packed_x, weights.w_gate,
                             weights.w_up, h, b.err, stream)
        B.moe_expert_down(self.desc, weights.inter, packed.region_offsets, h, weights.w_down, packed_y, b.err, stream)

    def expert_mlp_fp8(self, weights, packed: B.PackedBuffers, h: torch.Tensor, h_scales: torch.Tensor,
                       packed_y: torch.Tensor, stream=None):
        """The fp8 expert stage on e4m3 packed rows: linear 1 with SwiGLU into h
        (e4m3 [R*T*k][I]) and h_scales ([R*T*k][I/128]), then linear 2 into
        packed_y [R*T*k][H] bf16."""
        b = self.buf
        B.moe_expert_gate_up_fp8(self.desc, weights.inter, packed.region_offsets, packed.packed_x,
                                 packed.packed_scales, weights.w_gate, weights.w_gate_scales, weights.w_up,
                                 weights.w_up_scales, h, h_scales, b.err, stream)
        B.moe_expert_down_fp8(self.desc, weights.inter, packed.region_offsets, h, h_scales, weights.w_down,
                              weights.w_down_scales, packed_y, b.err, stream)

    def error(self, stream=None) -> int:
        return B.moe_get_error(self.buf.err, stream)
