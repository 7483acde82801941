"""Python binding of libmoe_layout.so: argument marshalling only.

Every function has the name of the C entry point it calls (see
include/moe_layout.h) and passes device pointers of torch tensors plus the
current CUDA stream; all the work runs in the library's kernels. There is no
fallback: if the library cannot be built or loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _build

MOE_OK, MOE_EINVAL, MOE_EOVERFLOW, MOE_ETIMEOUT, MOE_ECUDA, MOE_ENOMEM = 0, -1, -2, -3, -4, -5
MOE_BF16, MOE_FP8_E4M3, MOE_BF16_TO_FP8 = 0, 1, 2


class MoeDesc(ctypes.Structure):
    _fields_ = [
        ("num_ranks", ctypes.c_int32),
        ("tokens_per_rank", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("max_m", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
    ]

    @classmethod
    def of(cls, workload, num_sms: int = 0) -> "MoeDesc":
        w = workload
        return cls(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk, w.max_m, w.dtype_code, num_sms)


class MoeSizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("recv_x", "recv_scales", "recv_meta", "counts", "flags", "tok_slot", "expert_out")]


MOE_MAX_PARTS = 8


class MoeParts(ctypes.Structure):
    """The receive side in G parts (moe_parts of include/moe_layout.h)."""
    _fields_ = [
        ("num_parts", ctypes.c_int32),
        ("recv_x", ctypes.c_void_p * MOE_MAX_PARTS),
        ("recv_scales", ctypes.c_void_p * MOE_MAX_PARTS),
        ("recv_meta", ctypes.c_void_p * MOE_MAX_PARTS),
        ("flags", ctypes.c_void_p * MOE_MAX_PARTS),
        ("expert_out", ctypes.c_void_p * MOE_MAX_PARTS),
    ]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_status_string(status)} (status {status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Build (if stale) and open libmoe_layout.so; raises if that is impossible."""
    global _lib
    if _lib is None:
        _lib = _open(_build.build())
    return _lib


def _open(path: str):
    """Open a build of the library at `path` and declare its entry points."""
    lib = ctypes.CDLL(path)
    vp, st = ctypes.c_void_p, ctypes.c_int32
    pdesc = ctypes.POINTER(MoeDesc)
    lib.moe_buffer_sizes.argtypes = [pdesc, ctypes.POINTER(MoeSizes)]
    lib.moe_layout.argtypes = [pdesc] + [vp] * 6
    lib.moe_dispatch.argtypes = [pdesc] + [vp] * 9
    lib.moe_layout_dispatch.argtypes = [pdesc] + [vp] * 11
    lib.moe_dispatch_recv.argtypes = [pdesc] + [vp] * 13
    lib.moe_combine_packed.argtypes = [pdesc] + [vp] * 7
    lib.moe_route_stats.argtypes = [pdesc, vp, ctypes.c_int32, vp, vp, vp]
    lib.moe_expert_stub.argtypes = [pdesc] + [vp] * 6
    lib.moe_expert_gate_up.argtypes = [pdesc, ctypes.c_int32] + [vp] * 7
    lib.moe_expert_down.argtypes = [pdesc, ctypes.c_int32] + [vp] * 6
    lib.moe_expert_mlp_noalloc.argtypes = [pdesc, ctypes.c_int32] + [vp] * 8
    lib.moe_expert_mlp_noalloc_fp8.argtypes = [pdesc, ctypes.c_int32] + [vp] * 12
    lib.moe_expert_gate_up_fp8.argtypes = [pdesc, ctypes.c_int32] + [vp] * 11
    lib.moe_expert_down_fp8.argtypes = [pdesc, ctypes.c_int32] + [vp] * 8
    lib.moe_combine.argtypes = [pdesc] + [vp] * 7
    lib.moe_reset.argtypes = [pdesc] + [vp] * 3
    pparts = ctypes.POINTER(MoeParts)
    lib.moe_layout_dispatch_parts.argtypes = [pdesc, vp, vp, vp, vp, vp, pparts, vp, vp]
    lib.moe_combine_parts.argtypes = [pdesc, pparts, vp, vp, vp, vp, vp]
    lib.moe_expert_stub_parts.argtypes = [pdesc, pparts, vp, vp, vp]
    lib.moe_reset_parts.argtypes = [pdesc, pparts, vp, vp]
    lib.moe_get_error.argtypes = [vp, vp]
    lib.moe_layout_dispatch_kernels.argtypes = [pdesc]
    lib.moe_layout_dispatch_kernels.restype = ctypes.c_int32
    lib.moe_status_string.argtypes = [ctypes.c_int32]
    lib.moe_status_string.restype = ctypes.c_char_p
    for name in ("moe_buffer_sizes", "moe_layout", "moe_dispatch", "moe_layout_dispatch", "moe_dispatch_recv",
                 "moe_expert_stub", "moe_combine", "moe_combine_packed", "moe_route_stats", "moe_reset",
                 "moe_expert_gate_up", "moe_expert_down", "moe_expert_mlp_noalloc", "moe_expert_gate_up_fp8",
                 "moe_expert_down_fp8", "moe_expert_mlp_noalloc_fp8", "moe_layout_dispatch_parts",
                 "moe_combine_parts", "moe_expert_stub_parts", "moe_reset_parts", "moe_get_error"):
        getattr(lib, name).restype = st
    return lib


def _ptr(t: torch.Tensor | None, host_ok: bool = False):
    """Device pointer of a tensor; host_ok also admits pinned host memory (the
    step's inputs and output, which the kernels can read and write directly)."""
    if t is None:
        return None
    if not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError("libmoe_layout takes device tensors" + (" or pinned host tensors" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError("libmoe_layout takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_buffer_sizes(desc: MoeDesc) -> dict:
    out = MoeSizes()
    _check(load().moe_buffer_sizes(ctypes.byref(desc), ctypes.byref(out)), "moe_buffer_sizes")
    return {name: int(getattr(out, name)) for name, _ in MoeSizes._fields_}


def moe_layout(desc, topk_idx, counts, flags, tok_slot, err, stream=None):
    _check(load().moe_layout(ctypes.byref(desc), _ptr(topk_idx, True), _ptr(counts), _ptr(flags), _ptr(tok_slot),
                             _ptr(err), _stream(stream)), "moe_layout")


def moe_dispatch(desc, x, x_scales, tok_slot, flags, recv_x, recv_scales, recv_meta, err, stream=None):
    _check(load().moe_dispatch(ctypes.byref(desc), _ptr(x, True), _ptr(x_scales, True), _ptr(tok_slot), _ptr(flags),
                               _ptr(recv_x), _ptr(recv_scales), _ptr(recv_meta), _ptr(err), _stream(stream)),
           "moe_dispatch")


def moe_layout_dispatch(desc, topk_idx, x, x_scales, counts, flags, tok_slot, recv_x, recv_scales, recv_meta, err,
                        stream=None):
    _check(load().moe_layout_dispatch(ctypes.byref(desc), _ptr(topk_idx, True), _ptr(x, True), _ptr(x_scales, True),
                                      _ptr(counts),
                                      _ptr(flags), _ptr(tok_slot), _ptr(recv_x), _ptr(recv_scales), _ptr(recv_meta),
                                      _ptr(err), _stream(stream)), "moe_layout_dispatch")


def moe_layout_dispatch_kernels(desc) -> int:
    n = int(load().moe_layout_dispatch_kernels(ctypes.byref(desc)))
    _check(min(n, 0), "moe_layout_dispatch_kernels")
    return n


def moe_expert_stub(desc, recv_x, recv_scales, counts, expert_out, err, stream=None):
    _check(load().moe_expert_stub(ctypes.byref(desc), _ptr(recv_x), _ptr(recv_scales), _ptr(counts),
                                  _ptr(expert_out), _ptr(err), _stream(stream)), "moe_expert_stub")


def moe_expert_gate_up(desc, inter: int, region_offsets, packed_x, w_gate, w_up, h, err, stream=None):
    _check(load().moe_expert_gate_up(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(packed_x),
                                     _ptr(w_gate), _ptr(w_up), _ptr(h), _ptr(err), _stream(stream)),
           "moe_expert_gate_up")


def moe_expert_down(desc, inter: int, region_offsets, h, w_down, packed_y, err, stream=None):
    _check(load().moe_expert_down(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(h), _ptr(w_down),
                                  _ptr(packed_y), _ptr(err), _stream(stream)), "moe_expert_down")


def moe_expert_gate_up_fp8(desc, inter: int, region_offsets, packed_x, packed_scales, w_gate, w_gate_scales, w_up,
                           w_up_scales, h, h_scales, err, stream=None):
    _check(load().moe_expert_gate_up_fp8(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(packed_x),
                                         _ptr(packed_scales), _ptr(w_gate), _ptr(w_gate_scales), _ptr(w_up),
                                         _ptr(w_up_scales), _ptr(h), _ptr(h_scales), _ptr(err), _stream(stream)),
           "moe_expert_gate_up_fp8")


def moe_expert_down_fp8(desc, inter: int, region_offsets, h, h_scales, w_down, w_down_scales, packed_y, err,
                        stream=None):
    _check(load().moe_expert_down_fp8(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(h), _ptr(h_scales),
                                      _ptr(w_down), _ptr(w_down_scales), _ptr(packed_y), _ptr(err), _stream(stream)),
           "moe_expert_down_fp8")


def moe_expert_mlp_noalloc(desc, inter: int, region_offsets, packed_x, w_gate, w_up, w_down, packed_y, err,
                           stream=None):
    _check(load().moe_expert_mlp_noalloc(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(packed_x),
                                         _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(packed_y), _ptr(err),
                                         _stream(stream)), "moe_expert_mlp_noalloc")


def moe_expert_mlp_noalloc_fp8(desc, inter: int, region_offsets, packed_x, packed_scales, w_gate, w_gate_scales,
                               w_up, w_up_scales, w_down, w_down_scales, packed_y, err, stream=None):
    _check(load().moe_expert_mlp_noalloc_fp8(ctypes.byref(desc), int(inter), _ptr(region_offsets), _ptr(packed_x),
                                             _ptr(packed_scales), _ptr(w_gate), _ptr(w_gate_scales), _ptr(w_up),
                                             _ptr(w_up_scales), _ptr(w_down), _ptr(w_down_scales), _ptr(packed_y),
                                             _ptr(err), _stream(stream)), "moe_expert_mlp_noalloc_fp8")


def moe_combine(desc, expert_out, topk_weights, tok_slot, flags, out, err, stream=None):
    _check(load().moe_combine(ctypes.byref(desc), _ptr(expert_out), _ptr(topk_weights, True), _ptr(tok_slot),
                              _ptr(flags), _ptr(out, True), _ptr(err), _stream(stream)), "moe_combine")


def moe_dispatch_recv(desc, counts, flags, recv_x, recv_scales, recv_meta, tok_slot, region_offsets, packed_x,
                      packed_scales, packed_meta, tok_packed, err, stream=None):
    _check(load().moe_dispatch_recv(ctypes.byref(desc), _ptr(counts), _ptr(flags), _ptr(recv_x), _ptr(recv_scales),
                                    _ptr(recv_meta), _ptr(tok_slot), _ptr(region_offsets), _ptr(packed_x),
                                    _ptr(packed_scales), _ptr(packed_meta), _ptr(tok_packed), _ptr(err),
                                    _stream(stream)),
           "moe_dispatch_recv")


def moe_combine_packed(desc, packed_y, tok_packed, topk_weights, flags, out, err, stream=None):
    _check(load().moe_combine_packed(ctypes.byref(desc), _ptr(packed_y), _ptr(tok_packed), _ptr(topk_weights, True),
                                     _ptr(flags), _ptr(out, True), _ptr(err), _stream(stream)), "moe_combine_packed")


def moe_route_stats(desc, topk_idx, ranks_per_node: int, stats, err, stream=None):
    _check(load().moe_route_stats(ctypes.byref(desc), _ptr(topk_idx, True), int(ranks_per_node), _ptr(stats),
                                  _ptr(err), _stream(stream)), "moe_route_stats")


def moe_reset(desc, flags, err, stream=None):
    _check(load().moe_reset(ctypes.byref(desc), _ptr(flags), _ptr(err), _stream(stream)), "moe_reset")


def moe_layout_dispatch_parts(desc, topk_idx, x, x_scales, counts, tok_slot, parts: "PartBuffers", err,
                              stream=None):
    _check(load().moe_layout_dispatch_parts(ctypes.byref(desc), _ptr(topk_idx, True), _ptr(x, True),
                                            _ptr(x_scales, True), _ptr(counts), _ptr(tok_slot),
                                            ctypes.byref(parts.table()), _ptr(err), _stream(stream)),
           "moe_layout_dispatch_parts")


def moe_combine_parts(desc, parts: "PartBuffers", topk_weights, tok_slot, out, err, stream=None):
    _check(load().moe_combine_parts(ctypes.byref(desc), ctypes.byref(parts.table()), _ptr(topk_weights, True),
                                    _ptr(tok_slot), _ptr(out, True), _ptr(err), _stream(stream)), "moe_combine_parts")


def moe_expert_stub_parts(desc, parts: "PartBuffers", counts, err, stream=None):
    _check(load().moe_expert_stub_parts(ctypes.byref(desc), ctypes.byref(parts.table()), _ptr(counts), _ptr(err),
                                        _stream(stream)), "moe_expert_stub_parts")


def moe_reset_parts(desc, parts: "PartBuffers", err, stream=None):
    _check(load().moe_reset_parts(ctypes.byref(desc), ctypes.byref(parts.table()), _ptr(err), _stream(stream)),
           "moe_reset_parts")


def moe_get_error(err, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns its status code."""
    return int(load().moe_get_error(_ptr(err), _stream(stream)))


@dataclass
class MoeBuffers:
    """Device buffers of one step, sized by moe_buffer_sizes (allocated with torch)."""
    counts: torch.Tensor
    flags: torch.Tensor
    tok_slot: torch.Tensor
    recv_x: torch.Tensor
    recv_scales: torch.Tensor | None
    recv_meta: torch.Tensor
    expert_out: torch.Tensor | None
    out: torch.Tensor
    err: torch.Tensor


@dataclass
class PackedBuffers:
    """Outputs of moe_dispatch_recv: expert-major rows of the filled slots."""
    region_offsets: torch.Tensor  # [E*R + 1] int32
    packed_x: torch.Tensor        # [R*T*k, row bytes] uint8
    packed_scales: torch.Tensor | None
    packed_meta: torch.Tensor     # [R*T*k, 4] int32
    tok_packed: torch.Tensor      # [R, T, k] int32


def allocate_packed(desc: MoeDesc, device) -> PackedBuffers:
    R, T, H, E, k = desc.num_ranks, desc.tokens_per_rank, desc.hidden, desc.num_experts, desc.topk
    n = max(1, R * T * k)
    row = 2 * H if desc.dtype == MOE_BF16 else H
    dev = torch.device(device)
    return PackedBuffers(
        region_offsets=torch.zeros(E * R + 1, dtype=torch.int32, device=dev),
        packed_x=torch.empty((n, row), dtype=torch.uint8, device=dev),
        packed_scales=torch.empty((n, H // 128), dtype=torch.float32, device=dev) if desc.dtype != MOE_BF16 else None,
        packed_meta=torch.empty((n, 4), dtype=torch.int32, device=dev),
        tok_packed=torch.empty((R, T, k), dtype=torch.int32, device=dev),
    )


def allocate_buffers(desc: MoeDesc, device, with_expert_out: bool | None = None) -> MoeBuffers:
    """Allocate every buffer of a step. expert_out is allocated for fp8 steps
    (identity experts of bf16 steps read recv_x directly) unless overridden."""
    sz = moe_buffer_sizes(desc)
    R, T, H, E, k, M = desc.num_ranks, desc.tokens_per_rank, desc.hidden, desc.num_experts, desc.topk, desc.max_m
    slots = E * R * M
    fp8 = desc.dtype != MOE_BF16  # slots hold e4m3 rows + scales
    dev = torch.device(device)
    recv_x = torch.empty(sz["recv_x"], dtype=torch.uint8, device=dev).view(slots, -1)
    recv_scales = torch.empty((slots, H // 128), dtype=torch.float32, device=dev) if fp8 else None
    if with_expert_out is None:
        with_expert_out = fp8
    expert_out = torch.empty((slots, H), dtype=torch.bfloat16, device=dev) if with_expert_out else None
    return MoeBuffers(
        counts=torch.zeros((E, R), dtype=torch.int32, device=dev),
        flags=torch.zeros((E, R), dtype=torch.int64, device=dev),  # uint64 count+1 words
        tok_slot=torch.empty((R, T, k), dtype=torch.int32, device=dev),
        recv_x=recv_x,
        recv_scales=recv_scales,
        recv_meta=torch.empty((slots, 4), dtype=torch.int32, device=dev),
        expert_out=expert_out,
        out=torch.empty((R, T, H), dtype=torch.bfloat16, device=dev),
        err=torch.zeros(1, dtype=torch.int32, device=dev),
    )


@dataclass
class PartBuffers:
    """The receive side in G parts: part g holds the regions of ranks
    [g*R/G, (g+1)*R/G), every buffer 1/G of moe_buffer_sizes' size."""
    recv_x: list
    recv_scales: list | None
    recv_meta: list
    flags: list
    expert_out: list | None

    @property
    def num_parts(self) -> int:
        return len(self.recv_x)

    def table(self) -> MoeParts:
        t = MoeParts()
        t.num_parts = self.num_parts
        for g in range(self.num_parts):
            t.recv_x[g] = _ptr(self.recv_x[g]).value
            t.recv_meta[g] = _ptr(self.recv_meta[g]).value
            t.flags[g] = _ptr(self.flags[g]).value
            if self.recv_scales is not None:
                t.recv_scales[g] = _ptr(self.recv_scales[g]).value
            if self.expert_out is not None:
                t.expert_out[g] = _ptr(self.expert_out[g]).value
        return t


def allocate_parts(desc: MoeDesc, num_parts: int, device, with_expert_out: bool | None = None,
                   alloc=None) -> PartBuffers:
    """Separate allocations for each part of the receive side. alloc(shape,
    dtype) makes one buffer (default torch.empty on the device)."""
    R, H, E, M = desc.num_ranks, desc.hidden, desc.num_experts, desc.max_m
    if num_parts < 1 or num_parts > MOE_MAX_PARTS or R % num_parts:
        raise ValueError("num_parts must divide the ranks and be at most MOE_MAX_PARTS")
    dev = torch.device(device)
    if alloc is None:
        def alloc(shape, dtype):
            return torch.empty(shape, dtype=dtype, device=dev)
    slots = E * R * M // num_parts
    regions = E * R // num_parts
    fp8 = desc.dtype != MOE_BF16
    row = H if fp8 else 2 * H
    if with_expert_out is None:
        with_expert_out = fp8
    G = range(num_parts)
    return PartBuffers(
        recv_x=[alloc((slots, row), torch.uint8) for _ in G],
        recv_scales=[alloc((slots, H // 128), torch.float32) for _ in G] if fp8 else None,
        recv_meta=[alloc((slots, 4), torch.int32) for _ in G],
        flags=[alloc((regions,), torch.int64) for _ in G],
        expert_out=[alloc((slots, H), torch.bfloat16) for _ in G] if with_expert_out else None,
    )
